// Planner: turns the batch metadata into the work lists of the two
// attention kernels, on the device, once per pa_attention call.
//
//  - Requests with at least kPrefillMinQlen new tokens become tensor-core
//    work items (two 128-row tiles of one kv head each), bucket-sorted by the
//    number of 64-key tiles they read, longest first.
//  - Every other new token becomes a split-KV unit: the compacted list
//    {token, request, keys to attend, first flattened position} with the
//    prefix sum of Hkv * ceil(keys / 16) positions, which the split-KV
//    kernel's workers slice into equal parts.
//  - Cascade calls (common prefix of prefix_blocks blocks): every span goes
//    to the split-KV path with the prefix blocks left out of its positions;
//    requests must see the whole prefix and start with request 0's prefix
//    blocks, which is checked here.
// Invalid spans or lengths are skipped and reported on the device error word.
// A decode-only batch needs no planner: the split-KV kernel builds its own
// unit list.
#include "pa_internal.h"
#include "ptx.cuh"

namespace pa {

constexpr unsigned kFull = 0xffffffffu;

constexpr int kPlanThreads = 1024;

__device__ __forceinline__ long long block_exclusive_scan(long long v, long long* total,
                                                          long long* sm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  long long x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long y = __shfl_up_sync(kFull, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sm[warp] = x;
  __syncthreads();
  if (warp == 0) {
    long long s = lane < nw ? sm[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(kFull, s, o);
      if (lane >= o) s += y;
    }
    sm[lane] = s;
  }
  __syncthreads();
  const long long before = warp ? sm[warp - 1] : 0;
  *total = sm[nw - 1];
  __syncthreads();
  return before + x - v;
}

constexpr int kTileBuckets = 512;  // tiles sorted by key-tile count, longest first

__global__ void __launch_bounds__(kPlanThreads) pa_plan_kernel(PlanParams p) {
  // When the next grid has work that needs no plan (the cascade prefix
  // pass), let it start now; a grid that would only wait at its top for the
  // plan is released at the end of this one instead (starting it early
  // measured slower).
  if (p.early_trigger) griddep_launch_dependents();
  __shared__ long long scan_sm[32];
  __shared__ int bucket_cnt[kTileBuckets];
  __shared__ int bucket_pos[kTileBuckets];
  __shared__ int s_steps;    // prefill steps (item x key tile) of the batch
  __shared__ int s_workers;  // split-KV workers the slicing uses
  // Per-token scratch: {request, keys to attend}, then the compacted units'
  // first positions. In shared memory when the batch fits, else in the
  // workspace.
  extern __shared__ int2 dsm[];
  const int T = p.num_tokens;
  const bool in_smem = T <= kPlanSmemTokens;
  int2* const raw = in_smem ? dsm : p.raw;
  int* const ubase = in_smem ? reinterpret_cast<int*>(dsm + T) : nullptr;
  // a prefill work item is a pair of 128-row tiles: 2 * 128 / G chunk tokens
  const int tok_per_item = 2 * (128 / p.group);
  if (p.use_prefill)
    for (int b = threadIdx.x; b < kTileBuckets; b += blockDim.x) bucket_cnt[b] = 0;
  for (int t = threadIdx.x; t < T; t += blockDim.x) raw[t] = make_int2(-1, 0);
  if (threadIdx.x == 0) s_steps = 0;
  __syncthreads();

  // a request is valid when its span lies in [0, T] and its lengths agree
  // (the three loads are issued together: one DRAM round trip, not two)
  auto check = [&](int r, int& q0, int& qlen, int& L, bool report) -> bool {
    q0 = __ldg(p.qsl + r);
    const int q1 = __ldg(p.qsl + r + 1);
    L = __ldg(p.seq_lens + r);
    if (q0 < 0 || q1 < q0 || q1 > T) {
      if (report) report_error(p.err, PA_DEVERR_QSL, r);
      return false;
    }
    qlen = q1 - q0;
    if (L < qlen || (L + kBlockSize - 1) / kBlockSize > p.max_blocks_per_req ||
        qlen > p.max_query_len || L > p.max_seq_len ||
        L - qlen < p.prefix_blocks * kBlockSize) {
      if (report) report_error(p.err, PA_DEVERR_LENGTHS, r);
      return false;
    }
    return true;
  };
  auto tile_nkv = [&](int L, int ctx, int j0) -> int {  // 128-key tiles the item needs
    const int last = min(L - 1, ctx + j0 + tok_per_item - 1);  // last key of the item's rows
    return last / 128 + 1;
  };

  if (p.prefix_blocks > 0) {  // every table starts with request 0's prefix blocks
    // kCheckBatch independent loads per thread before any compare: one DRAM
    // round trip per batch rather than one per entry
    constexpr int kCheckBatch = 8;
    const long long n = (long long)(p.num_reqs - 1) * p.prefix_blocks;
    for (long long i0 = threadIdx.x; i0 < n; i0 += (long long)kCheckBatch * blockDim.x) {
      int got[kCheckBatch], want[kCheckBatch];
#pragma unroll
      for (int k = 0; k < kCheckBatch; ++k) {
        const long long i = i0 + (long long)k * blockDim.x;
        got[k] = want[k] = 0;
        if (i < n) {
          const int r = 1 + (int)(i / p.prefix_blocks), b = (int)(i % p.prefix_blocks);
          got[k] = __ldg(p.block_tables + (size_t)r * p.max_blocks_per_req + b);
          want[k] = __ldg(p.block_tables + b);
        }
      }
#pragma unroll
      for (int k = 0; k < kCheckBatch; ++k)
        if (got[k] != want[k])
          report_error(p.err, PA_DEVERR_PREFIX,
                       1 + (int)((i0 + (long long)k * blockDim.x) / p.prefix_blocks));
    }
  }
  for (int r = threadIdx.x; r < p.num_reqs; r += blockDim.x) {
    int q0, qlen, L;
    if (!check(r, q0, qlen, L, true)) continue;
    const int ctx = L - qlen;
    if (p.use_prefill && qlen >= kPrefillMinQlen) {
      int steps = 0;
      for (int j0 = 0; j0 < qlen; j0 += tok_per_item) {
        const int nkv = tile_nkv(L, ctx, j0);
        atomicAdd(&bucket_cnt[min(nkv, kTileBuckets - 1)], p.num_kv_heads);
        steps += nkv;
      }
      if (p.overlap) atomicAdd(&s_steps, steps * p.num_kv_heads);
      continue;  // these tokens are not on the split-KV path
    }
    for (int j = 0; j < qlen; ++j) raw[q0 + j] = make_int2(r, ctx + j + 1);
  }
  __syncthreads();
  if (p.use_prefill) {  // positions of the buckets, longest tiles first (exclusive scan, descending)
    static_assert(kTileBuckets <= kPlanThreads, "one bucket per thread");
    const int b = kTileBuckets - 1 - (int)threadIdx.x;  // blockDim is kPlanThreads here
    long long total;
    const long long ex = block_exclusive_scan(b >= 0 ? bucket_cnt[b] : 0, &total, scan_sm);
    if (b >= 0) bucket_pos[b] = (int)ex;
    if (threadIdx.x == 0) p.header->num_tiles = (int)total;
  } else if (threadIdx.x == 0) {
    p.header->num_tiles = 0;
  }
  __syncthreads();
  if (p.use_prefill) {
    for (int r = threadIdx.x; r < p.num_reqs; r += blockDim.x) {
      int q0, qlen, L;
      if (!check(r, q0, qlen, L, false) || qlen < kPrefillMinQlen) continue;
      const int ctx = L - qlen;
      for (int j0 = 0; j0 < qlen; j0 += tok_per_item) {
        const int nkv = tile_nkv(L, ctx, j0);
        const int at = atomicAdd(&bucket_pos[min(nkv, kTileBuckets - 1)], p.num_kv_heads);
        for (int kv = 0; kv < p.num_kv_heads; ++kv) p.tiles[at + kv] = PrefillTile{r, kv, j0, nkv};
      }
    }
  }
  // compaction: tokens with keys become units with their first flattened position
  constexpr long long kLow = (1LL << 40) - 1;
  long long run_k = 0, run_w = 0;
  for (int c0 = 0; c0 < T; c0 += blockDim.x) {
    const int t = c0 + threadIdx.x;
    const int2 u = t < T ? raw[t] : make_int2(-1, 0);
    // blocks on the split-KV path: all the token sees, less a cascade prefix
    const int nb = max(0, (u.y + kBlockSize - 1) / kBlockSize - p.prefix_blocks);
    // (token-major split-KV: one position per block, every kv head at once)
    const long long packed =
        ((long long)(nb > 0) << 40) | ((long long)nb * (p.token_major ? 1 : p.num_kv_heads));
    long long total;
    const long long ex = block_exclusive_scan(packed, &total, scan_sm);  // syncs: raw reads done
    if (nb > 0) {
      const int k = (int)(run_k + (ex >> 40));
      const int base = (int)(run_w + (ex & kLow));
      p.units[k] = UnitInfo{t, u.x, u.y, base};
      if (ubase) ubase[k] = base;
    }
    run_k += total >> 40;
    run_w += total & kLow;
  }
  const int K = (int)run_k, W = (int)run_w;
  if (threadIdx.x == 0) {
    p.units[K] = UnitInfo{T, -1, 0, W};  // base[K] = W
    if (ubase) ubase[K] = W;
    p.header->num_units = K;
    p.header->num_positions = W;
    // Overlapped mixed batch: the fewest SMs c that finish the prefill steps
    // (a margin ahead of) the split-KV work on the other S - c, if that beats
    // running the two one after the other. The split-KV time on n SMs is
    // bytes / min(n x per-SM rate, copy peak); the chunks alone on every SM
    // end at about 1.6x their even share (the longest items set the end).
    int ctas = p.num_sms, workers = p.num_workers;
    if (p.overlap && p.use_prefill && W > 0 && s_steps > 0) {
      const int S_ = p.num_sms;
      const float pre = kPrefillStepUs * (float)s_steps;  // SM x us
      const float bytes = (float)W * (float)p.position_bytes;
      auto dec_us = [&](int n) {
        return fmaxf(bytes / ((float)n * kDecodeSmBytesPerUs), bytes / kHbmBytesPerUs);
      };
      // smallest c with pre / c <= margin x dec_us(S - c), per branch of the max
      const float c1 = pre * (float)S_ * kDecodeSmBytesPerUs /
                       (kOverlapMargin * bytes + pre * kDecodeSmBytesPerUs);
      const float c2 = pre * kHbmBytesPerUs / (kOverlapMargin * bytes);
      const int c = max(1, (int)ceilf(fminf(fminf(c1, c2), (float)S_)));
      const float serial = 1.6f * pre / (float)S_ + dec_us(S_);
      if (p.prefill_ctas_override > 0) {  // the caller's share (at most half the SMs)
        ctas = min(p.prefill_ctas_override, S_ / 2);
        workers = min(workers, S_ - ctas);
      } else if (c <= S_ / 4 && dec_us(S_ - c) < serial) {
        ctas = c;
        workers = min(workers, S_ - c);
      }
    }
    p.header->prefill_ctas = ctas;
    p.header->decode_workers = workers;
    s_workers = workers;
  }
  // each split-KV worker's first unit (same worker count and slicing as the
  // split-KV kernel), found by binary search over the units' first positions
  __syncthreads();
  if (ubase) {
    const int NW = plan_workers(W, s_workers);
    for (int w = threadIdx.x; w < NW; w += blockDim.x) {
      const int S = (int)((long long)w * W / NW);
      int lo = 0, hi = K;  // ubase[lo] <= S < ubase[hi]
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (ubase[mid] <= S) lo = mid; else hi = mid;
      }
      p.worker_unit[w] = lo;
    }
  }
  // Let the grid before this one (the KV write on the same stream) finish
  // before this grid completes: whoever waits on the plan then also sees the
  // newly written K/V.
  if (!p.early_trigger) griddep_launch_dependents();
  griddep_wait();
}

cudaError_t launch_plan(const PlanParams& p, cudaStream_t s) {
  const int smem = p.num_tokens <= kPlanSmemTokens
                       ? (int)(sizeof(int2) * p.num_tokens + sizeof(int) * (p.num_tokens + 1))
                       : 0;
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    e = cudaFuncSetAttribute(pa_plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)(sizeof(int2) * kPlanSmemTokens + sizeof(int) * (kPlanSmemTokens + 1)));
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  // Launched as a programmatic dependent of the previous grid (normally the
  // KV write): it needs none of its output and overlaps it, and waits for it
  // before completing.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  // A batch with no tensor-core work needs no bucket sort: a block sized to the
  // batch (fewer warps per barrier) plans it faster.
  int threads = kPlanThreads;
  if (!p.use_prefill) {
    int need = p.num_tokens > p.num_reqs ? p.num_tokens : p.num_reqs;
    // a cascade's prefix check reads (requests - 1) x prefix blocks entries
    if (p.prefix_blocks > 0 && (long long)(p.num_reqs - 1) * p.prefix_blocks > need)
      need = kPlanThreads;
    threads = need <= 128 ? 128 : need <= 256 ? 256 : need <= 512 ? 512 : kPlanThreads;
  }
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, pa_plan_kernel, p);
}

}  // namespace pa
