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
//  - The merge counters of every (unit, kv head) are zeroed.
// Invalid spans or lengths are skipped and reported on the device error word.
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
  // The dependent grid may be scheduled now; it waits for this grid to
  // finish before reading the plan.
  griddep_launch_dependents();
  __shared__ long long scan_sm[32];
  __shared__ int bucket_cnt[kTileBuckets];
  __shared__ int bucket_pos[kTileBuckets];
  const int T = p.num_tokens;
  // a prefill work item is a pair of 128-row tiles: 2 * 128 / G chunk tokens
  const int tok_per_item = 2 * (128 / p.group);
  for (int b = threadIdx.x; b < kTileBuckets; b += blockDim.x) bucket_cnt[b] = 0;
  for (int t = threadIdx.x; t < T; t += blockDim.x) p.units[t] = UnitInfo{t, -1, 0, 0};
  __syncthreads();

  // a request is valid when its span lies in [0, T] and its lengths agree
  auto check = [&](int r, int& q0, int& qlen, int& L, bool report) -> bool {
    q0 = p.qsl[r];
    const int q1 = p.qsl[r + 1];
    if (q0 < 0 || q1 < q0 || q1 > T) {
      if (report) report_error(p.err, PA_DEVERR_QSL, r);
      return false;
    }
    qlen = q1 - q0;
    L = p.seq_lens[r];
    if (L < qlen || (L + kBlockSize - 1) / kBlockSize > p.max_blocks_per_req ||
        qlen > p.max_query_len || L > p.max_seq_len) {
      if (report) report_error(p.err, PA_DEVERR_LENGTHS, r);
      return false;
    }
    return true;
  };
  auto tile_nkv = [&](int L, int ctx, int j0) -> int {  // 128-key tiles the item needs
    const int last = min(L - 1, ctx + j0 + tok_per_item - 1);  // last key of the item's rows
    return last / 128 + 1;
  };

  for (int r = threadIdx.x; r < p.num_reqs; r += blockDim.x) {
    int q0, qlen, L;
    if (!check(r, q0, qlen, L, true)) continue;
    const int ctx = L - qlen;
    if (p.use_prefill && qlen >= kPrefillMinQlen) {
      for (int j0 = 0; j0 < qlen; j0 += tok_per_item)
        atomicAdd(&bucket_cnt[min(tile_nkv(L, ctx, j0), kTileBuckets - 1)], p.num_kv_heads);
      continue;  // these tokens are not on the split-KV path
    }
    for (int j = 0; j < qlen; ++j) p.units[q0 + j] = UnitInfo{q0 + j, r, ctx + j + 1, 0};
  }
  __syncthreads();
  {  // positions of the buckets, longest tiles first (exclusive scan, descending)
    static_assert(kTileBuckets <= kPlanThreads, "one bucket per thread");
    const int b = kTileBuckets - 1 - (int)threadIdx.x;
    long long total;
    const long long ex = block_exclusive_scan(b >= 0 ? bucket_cnt[b] : 0, &total, scan_sm);
    if (b >= 0) bucket_pos[b] = (int)ex;
    if (threadIdx.x == 0) p.header->num_tiles = (int)total;
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
  __syncthreads();
  constexpr long long kLow = (1LL << 40) - 1;
  long long run_k = 0, run_w = 0;
  for (int c0 = 0; c0 < T; c0 += blockDim.x) {
    const int t = c0 + threadIdx.x;
    const UnitInfo u = t < T ? p.units[t] : UnitInfo{0, -1, 0, 0};
    const int nb = (u.len + kBlockSize - 1) / kBlockSize;
    const long long packed = ((long long)(nb > 0) << 40) | ((long long)nb * p.num_kv_heads);
    long long total;
    const long long ex = block_exclusive_scan(packed, &total, scan_sm);
    if (nb > 0) p.units[run_k + (ex >> 40)] = UnitInfo{u.tok, u.req, u.len, (int)(run_w + (ex & kLow))};
    run_k += total >> 40;
    run_w += total & kLow;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    p.units[run_k] = UnitInfo{T, -1, 0, (int)run_w};  // base[K] = W
    p.header->num_units = (int)run_k;
    p.header->num_positions = (int)run_w;
  }
  for (long long i = threadIdx.x; i < run_k * p.num_kv_heads; i += blockDim.x) p.counters[i] = 0;
}

cudaError_t launch_plan(const PlanParams& p, cudaStream_t s) {
  pa_plan_kernel<<<1, kPlanThreads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace pa
