// KV-cache write: scatter each new token's K and V rows into its physical
// slot ("vLLM v1 Deep Dive: How LLM(...) and the Server Boot and Generate",
// Part 3, "Aside - KV cache and prefix caching": the slot is
// block_id * block_size + offset and the scatter is phase-agnostic - a prefill
// token and a decode token are written the same way).
//
// Cache layout [num_blocks][Hkv][16][D]: the destination of (token t, head h)
// is one contiguous D-element row. The kernel is a pure copy: each thread moves
// one 16-byte vector of K and the matching vector of V, so a warp covers two
// (D=128) or four (D=64) full rows with fully coalesced 128-bit loads and
// stores. Bandwidth-bound, no shared memory.
#include "pa_internal.h"
#include "ptx.cuh"

namespace pa {

__global__ void __launch_bounds__(256) pa_write_kv_kernel(WriteParams p) {
  // A planner launched next may start now: it reads only metadata, and
  // waits for this grid before it completes.
  griddep_launch_dependents();
  const int vec_per_row = p.head_dim / 8;  // 16-byte vectors per D-element row
  const long long total = (long long)p.num_tokens * p.num_kv_heads * vec_per_row;
  const uint4* k = reinterpret_cast<const uint4*>(p.k);
  const uint4* v = reinterpret_cast<const uint4*>(p.v);
  uint4* kc = reinterpret_cast<uint4*>(p.k_cache);
  uint4* vc = reinterpret_cast<uint4*>(p.v_cache);
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const long long row = i / vec_per_row;  // t * Hkv + h
    const int c = (int)(i - row * vec_per_row);
    const int t = (int)(row / p.num_kv_heads);
    const int h = (int)(row - (long long)t * p.num_kv_heads);
    const long long s = __ldg(p.slot_mapping + t);
    if (s < 0) continue;  // padding token
    if (s >= p.num_slots) {
      report_error(p.err, PA_DEVERR_SLOT, t);
      continue;
    }
    const long long blk = s >> 4, off = s & 15;
    const long long dst = ((blk * p.num_kv_heads + h) * kBlockSize + off) * vec_per_row + c;
    const uint4 kv = __ldg(k + i);
    const uint4 vv = __ldg(v + i);
    kc[dst] = kv;
    vc[dst] = vv;
  }
}

// FP8 cache ("vLLM: An Exhaustive Technical Study for Kernel Engineers", 2.8:
// --kv-cache-dtype fp8 is E4M3 with an fp32 per-tensor scale): the same
// scatter, each element stored as E4M3(x / scale). The quotient is a
// correctly rounded binary32 division; the conversion rounds to nearest even
// and saturates at +-448. A thread turns 8 bf16 values (16 bytes) into 8
// codes (8 bytes).
__global__ void __launch_bounds__(256) pa_write_kv_fp8_kernel(WriteParams p) {
  griddep_launch_dependents();
  const int vec_per_row = p.head_dim / 8;
  const long long total = (long long)p.num_tokens * p.num_kv_heads * vec_per_row;
  const uint4* k = reinterpret_cast<const uint4*>(p.k);
  const uint4* v = reinterpret_cast<const uint4*>(p.v);
  uint2* kc = reinterpret_cast<uint2*>(p.k_cache);
  uint2* vc = reinterpret_cast<uint2*>(p.v_cache);
  auto quant = [](uint4 x, float s) -> uint2 {
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
    uint32_t o[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const float2 a = bf16x2_to_float2(w[2 * i]);
      const float2 b = bf16x2_to_float2(w[2 * i + 1]);
      const uint16_t ca = float2_to_e4m3x2(__fdiv_rn(a.x, s), __fdiv_rn(a.y, s));
      const uint16_t cb = float2_to_e4m3x2(__fdiv_rn(b.x, s), __fdiv_rn(b.y, s));
      o[i] = (uint32_t)ca | ((uint32_t)cb << 16);
    }
    return make_uint2(o[0], o[1]);
  };
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const long long row = i / vec_per_row;
    const int c = (int)(i - row * vec_per_row);
    const int t = (int)(row / p.num_kv_heads);
    const int h = (int)(row - (long long)t * p.num_kv_heads);
    const long long s = __ldg(p.slot_mapping + t);
    if (s < 0) continue;
    if (s >= p.num_slots) {
      report_error(p.err, PA_DEVERR_SLOT, t);
      continue;
    }
    const long long blk = s >> 4, off = s & 15;
    const long long dst = ((blk * p.num_kv_heads + h) * kBlockSize + off) * vec_per_row + c;
    kc[dst] = quant(__ldg(k + i), p.k_scale);
    vc[dst] = quant(__ldg(v + i), p.v_scale);
  }
}

cudaError_t launch_write_kv(const WriteParams& p, cudaStream_t s) {
  const long long total = (long long)p.num_tokens * p.num_kv_heads * (p.head_dim / 8);
  if (total == 0) return cudaSuccess;
  const int threads = 256;
  long long blocks = (total + threads - 1) / threads;
  if (blocks > 65535LL * 16) blocks = 65535LL * 16;
  if (p.kv_fp8)
    pa_write_kv_fp8_kernel<<<(unsigned)blocks, threads, 0, s>>>(p);
  else
    pa_write_kv_kernel<<<(unsigned)blocks, threads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace pa
