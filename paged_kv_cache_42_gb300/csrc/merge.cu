// Merge pass of the split-KV decode.
//
// The split-KV kernel gives each warp an equal slice of the flattened
// (token, kv head, 16-key block) positions. A (token, kv head) whose blocks
// fall into more than one slice leaves one unnormalised partial (m, l, o)
// per slice, in slots u + wf .. u + wl (u = token * Hkv + kv head, wf .. wl
// the workers whose slices hold its first and last block). This pass runs
// after the split-KV grid (chained by programmatic launch, it waits on that
// grid before reading) and combines them by log-sum-exp renormalisation
// ("vLLM: An Exhaustive Technical Study for Kernel Engineers", 2.3, the merge
// of partial attention states) in a fixed order of operations, so the result
// does not depend on which warp finished first. In a cascade call the prefix
// partials of the same (token, kv head) are merged in with the suffix slots.
//
// One CTA per slice boundary, reading the task the split-KV worker after the
// boundary left for it. Its warps split the partials between them, each
// merging its share online (the loads of the next partial are independent of
// the arithmetic), and combine their results through shared memory; so a
// merge takes about one round trip to L2 whatever the number of partials.
#include "pa_internal.h"
#include "ptx.cuh"

namespace pa {

namespace {

constexpr int kMergeWarps = 8;

template <int D, int G>
__global__ void __launch_bounds__(kMergeWarps * 32) pa_merge_kernel(const MergeParams p) {
  constexpr int V = D / 32;  // output dims per lane
  static_assert(V == 2 || V == 4, "head dim 64 or 128");
  __shared__ float s_m[kMergeWarps][G], s_l[kMergeWarps][G];
  __shared__ __align__(16) float s_o[kMergeWarps][G][D];
  griddep_wait();  // the split-KV grid's partials and tasks
  const int W = __ldcg(&p.header->num_positions);
  int nw = p.num_workers;
  if (p.workers_from_header) nw = min(nw, __ldcg(&p.header->decode_workers));
  if (W <= 0) return;
  int tok, kv, wf, wl;
  if (p.all_units) {
    // overlapped cascade: (unit, kv head) blockIdx; its positions, and the
    // workers holding them, as the split-KV kernel sliced them
    const int k = (int)blockIdx.x / p.num_kv_heads;
    kv = (int)blockIdx.x % p.num_kv_heads;
    if (k >= __ldcg(&p.header->num_units)) return;
    const int4 u = __ldcg(reinterpret_cast<const int4*>(p.units + k));
    const int nb = max(1, (u.z + kBlockSize - 1) / kBlockSize - p.key_start_blocks);
    const int first = u.w + kv * nb, NW = plan_workers(W, nw);
    tok = u.x;
    wf = worker_of(first, W, NW);
    wl = worker_of(first + nb - 1, W, NW);
  } else {
    const int w = (int)blockIdx.x + 1;
    const int4 task = __ldcg(p.tasks + w);
    // tasks past this call's worker count are stale
    if (w >= plan_workers(W, nw) || task.x < 0) return;
    tok = task.x;
    wf = task.z;
    wl = task.w;
    kv = task.y;
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

  // The partials: the suffix slots wf .. wl, then (cascade) the prefix chunks.
  // Worker wf + i's slot: u + wf + i (u = token * Hkv + kv head).
  const int u = tok * p.num_kv_heads + kv;
  const int ns = wl - wf + 1, n = ns + p.prefix_chunks;
  auto slot = [&](int i) -> const float* {
    const size_t s0 = (size_t)(u + wf + i);
    return i < ns ? p.partials + s0 * p.slot_floats
                  : p.prefix_partials +
                        (((size_t)(i - ns) * p.num_tokens + tok) * p.num_kv_heads + kv) *
                            p.slot_floats;
  };

  // this warp's share: partials warp, warp + kMergeWarps, ...
  float M[G], L[G], O[G][V];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    M[h] = -INFINITY;
    L[h] = 0.f;
#pragma unroll
    for (int i = 0; i < V; ++i) O[h][i] = 0.f;
  }
#pragma unroll 2
  for (int i = warp; i < n; i += kMergeWarps) {
    const float* sl = slot(i);
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float m = __ldcg(sl + h), l = __ldcg(sl + G + h);
      float o[V];
      if constexpr (V == 4) {
        const float4 v = __ldcg(reinterpret_cast<const float4*>(sl + 16 + h * D) + lane);
        o[0] = v.x;
        o[1] = v.y;
        o[2] = v.z;
        o[3] = v.w;
      } else {
        const float2 v = __ldcg(reinterpret_cast<const float2*>(sl + 16 + h * D) + lane);
        o[0] = v.x;
        o[1] = v.y;
      }
      const float mn = fmaxf(M[h], m);
      const float a = exp2f(M[h] - mn), b = exp2f(m - mn);  // M = -inf at first: a = 0
      L[h] = L[h] * a + l * b;
#pragma unroll
      for (int i2 = 0; i2 < V; ++i2) O[h][i2] = O[h][i2] * a + o[i2] * b;
      M[h] = mn;
    }
  }
#pragma unroll
  for (int h = 0; h < G; ++h) {
    if (lane == 0) {
      s_m[warp][h] = M[h];
      s_l[warp][h] = L[h];
    }
#pragma unroll
    for (int i = 0; i < V; ++i) s_o[warp][h][lane * V + i] = O[h][i];
  }
  __syncthreads();

  // combine the warps' shares (a warp without partials has m = -inf), two
  // output dims per thread, stored as one bf16 pair
  for (int e = threadIdx.x; e < G * D / 2; e += kMergeWarps * 32) {
    const int h = e / (D / 2), d = 2 * (e - h * (D / 2));
    float mx = -INFINITY;
#pragma unroll
    for (int k = 0; k < kMergeWarps; ++k) mx = fmaxf(mx, s_m[k][h]);
    float l = 0.f, o0 = 0.f, o1 = 0.f;
#pragma unroll
    for (int k = 0; k < kMergeWarps; ++k) {
      const float f = s_m[k][h] == -INFINITY ? 0.f : exp2f(s_m[k][h] - mx);
      l += s_l[k][h] * f;
      o0 += s_o[k][h][d] * f;
      o1 += s_o[k][h][d + 1] * f;
    }
    const float sc = p.v_scale / l;
    *reinterpret_cast<uint32_t*>(p.out + ((size_t)tok * p.num_q_heads + (size_t)kv * G + h) * D +
                                 d) = float2_to_bf16x2(o0 * sc, o1 * sc);
  }
}

// Token-major split-KV (eight KV heads): one CTA per slice boundary, one warp
// per KV head. A boundary's token leaves its partials in slots
// (token + w) * Hkv + kv for the workers w = wf .. wl that hold its blocks -
// usually two to a few dozen, so a warp merges its head's partials on its
// own, online, loading them a group at a time; no shared memory and no block
// barrier.
template <int D, int G>
__global__ void __launch_bounds__(kMergeWarps * 32) pa_merge_tm_kernel(const MergeParams p) {
  constexpr int V = D / 32;  // output dims per lane
  static_assert(V == 2 || V == 4, "head dim 64 or 128");
  griddep_wait();  // the split-KV grid's partials and tasks
  const int W = __ldcg(&p.header->num_positions);
  int nw = p.num_workers;
  if (p.workers_from_header) nw = min(nw, __ldcg(&p.header->decode_workers));
  if (W <= 0) return;
  const int w = (int)blockIdx.x + 1;
  const int4 task = __ldcg(p.tasks + w);
  if (w >= plan_workers(W, nw) || task.x < 0) return;  // stale task past this call's workers
  const int kv = (int)(threadIdx.x >> 5), lane = (int)(threadIdx.x & 31);
  if (kv >= p.num_kv_heads) return;
  const int tok = task.x, wf = task.z, n = task.w - task.z + 1;
  auto slot = [&](int i) -> const float* {
    return p.partials + ((size_t)(tok + wf + i) * p.num_kv_heads + kv) * p.slot_floats;
  };
  struct Part {
    float m[G], l[G], o[G][V];
  };
  auto load = [&](int i, Part& q) {
    const float* const sl = slot(i);
#pragma unroll
    for (int h = 0; h < G; ++h) {
      q.m[h] = __ldcg(sl + h);
      q.l[h] = __ldcg(sl + G + h);
      if constexpr (V == 4) {
        const float4 v = __ldcg(reinterpret_cast<const float4*>(sl + 16 + h * D) + lane);
        q.o[h][0] = v.x;
        q.o[h][1] = v.y;
        q.o[h][2] = v.z;
        q.o[h][3] = v.w;
      } else {
        const float2 v = __ldcg(reinterpret_cast<const float2*>(sl + 16 + h * D) + lane);
        q.o[h][0] = v.x;
        q.o[h][1] = v.y;
      }
    }
  };
  // partials in groups of K: a group's loads are all issued before any of
  // them is combined, so a group costs one round trip to L2
  constexpr int K = G <= 4 ? 4 : 2;
  Part acc, q[K];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    acc.m[h] = -INFINITY;
    acc.l[h] = 0.f;
#pragma unroll
    for (int e = 0; e < V; ++e) acc.o[h][e] = 0.f;
  }
  for (int i0 = 0; i0 < n; i0 += K) {
#pragma unroll
    for (int k = 0; k < K; ++k)
      if (i0 + k < n) load(i0 + k, q[k]);
#pragma unroll
    for (int k = 0; k < K; ++k) {
      if (i0 + k >= n) break;
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float mn = fmaxf(acc.m[h], q[k].m[h]);
        const float a = exp2f(acc.m[h] - mn), b = exp2f(q[k].m[h] - mn);  // acc.m = -inf: a = 0
        acc.l[h] = acc.l[h] * a + q[k].l[h] * b;
#pragma unroll
        for (int e = 0; e < V; ++e) acc.o[h][e] = acc.o[h][e] * a + q[k].o[h][e] * b;
        acc.m[h] = mn;
      }
    }
  }
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const float sc = p.v_scale / acc.l[h];
    uint16_t* const orow = p.out + ((size_t)tok * p.num_q_heads + (size_t)kv * G + h) * D;
    if constexpr (V == 4) {
      const uint2 pk = make_uint2(float2_to_bf16x2(acc.o[h][0] * sc, acc.o[h][1] * sc),
                                  float2_to_bf16x2(acc.o[h][2] * sc, acc.o[h][3] * sc));
      *reinterpret_cast<uint2*>(orow + lane * V) = pk;
    } else {
      *reinterpret_cast<uint32_t*>(orow + lane * V) =
          float2_to_bf16x2(acc.o[h][0] * sc, acc.o[h][1] * sc);
    }
  }
}

template <int D, int G>
cudaError_t launch_merge_t(const MergeParams& p, cudaStream_t s) {
  // one CTA per slice boundary, or per (token, kv head)
  const int boundaries = p.all_units ? p.num_tokens * p.num_kv_heads : p.num_workers - 1;
  if (boundaries <= 0) return cudaSuccess;  // one worker: nothing is ever split
  // token-major partials: eight KV heads, no cascade (the split-KV kernel's own limits)
  if (p.token_major && (p.all_units || p.prefix_chunks != 0 || p.num_kv_heads > kMergeWarps))
    return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)boundaries);
  cfg.blockDim = dim3(kMergeWarps * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  // Programmatic launch: the CTAs are placed as the split-KV grid's CTAs
  // retire and wait (griddepcontrol.wait) for the whole grid before reading.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (p.token_major) {  // a CTA per boundary, a warp per KV head
    cfg.blockDim = dim3(32 * p.num_kv_heads);
    return cudaLaunchKernelEx(&cfg, pa_merge_tm_kernel<D, G>, p);
  }
  return cudaLaunchKernelEx(&cfg, pa_merge_kernel<D, G>, p);
}

}  // namespace

cudaError_t launch_merge(const MergeParams& p, int head_dim, int group, cudaStream_t s) {
  if (head_dim == 128) {
    switch (group) {
      case 1: return launch_merge_t<128, 1>(p, s);
      case 2: return launch_merge_t<128, 2>(p, s);
      case 4: return launch_merge_t<128, 4>(p, s);
      case 8: return launch_merge_t<128, 8>(p, s);
    }
  } else if (head_dim == 64) {
    switch (group) {
      case 1: return launch_merge_t<64, 1>(p, s);
      case 2: return launch_merge_t<64, 2>(p, s);
      case 4: return launch_merge_t<64, 4>(p, s);
      case 8: return launch_merge_t<64, 8>(p, s);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace pa
