// Split-KV paged decode on the tensor cores (tcgen05 + TMEM + TMA).
//
// What is computed is exactly what the CUDA-core split-KV kernel (decode.cu)
// computes ("vLLM v1 Deep Dive: How LLM(...) and the Server Boot and
// Generate", Part 3, "Aside - KV cache and prefix caching": a decode query
// attends to all of its request's blocks, a token of a short span to keys
// 0 .. ctx + j; "vLLM: An Exhaustive Technical Study for Kernel Engineers",
// 2.4: the query heads sharing a KV head are processed together, so each K/V
// block is read once per KV head). It takes the same work list (the planner's
// units, or its own for a decode-only batch), the same flattened (token, kv
// head, 16-key block) positions sliced into equal contiguous parts, and
// leaves the same partial slots and merge tasks for the merge pass
// (merge.cu). Only the worker differs: one CTA instead of one warp.
//
// Why tensor cores. A cached K/V element is used by all G query heads of its
// group: 4G flops per 2-byte element. At G = 8 that arithmetic, on the FMA
// pipe, and not the HBM bytes, sets the pace of the CUDA-core kernel, and at
// G = 4 it balances the bytes. Here both contractions run on the tensor pipe,
// which leaves the CUDA cores the softmax alone.
//
// Formulation (ours). For a (token, kv head) and a tile of 128 keys (eight
// 16-key cache blocks):
//   S^T = K Q^T      tcgen05.mma kind::f16, M = 128 keys, N = 16 (the G query
//                    heads of the group, zero-padded), K = head_dim; A = the K
//                    tile and B = the G q rows, 128B-swizzled K-major in
//                    shared memory; fp32 into TMEM (lane = key).
//   softmax          one thread per key (its TMEM lane): mask, scale, the
//                    tile's max over 128 keys (warp shuffles, then a 4-warp
//                    exchange on an mbarrier), exp2; P^T rounded to bf16 into
//                    shared memory in the B-operand layout.
//   O^T += V^T P^T   M = 128 head dims, N = 16, K = 128 keys; A = the same V
//                    tile image read M/N-major, B = P^T; O^T stays in TMEM
//                    (lane = head dim) across the tiles of a (token, kv head),
//                    always accumulating: its columns start at zero and the
//                    epilogue of a portion zeroes them after reading them.
// The reference max moves (and O is rescaled through TMEM) only when a tile's
// max exceeds it by more than 2^8, so P <= 256 and the result stays exact up
// to rounding; with ordinary score spreads that happens only at a segment's
// first tile.
//
// Full tiles. A CTA's slice is cut into tiles of eight consecutive positions
// whatever the (token, kv head) boundaries: a tile may hold the end of one
// portion (a (token, kv head) part of the slice) and the start of the next.
// Portion n of the CTA takes slot n % 2, which is half of the MMA's N = 16:
// its q rows are rows 8 slot .. 8 slot + G - 1 of the N operand, its scores
// and outputs columns 8 slot .. of S^T and O^T, so one MMA pair serves both.
// Keeping tiles full keeps each CTA's bytes in flight, and so its share of
// HBM, independent of where its portions end: with one portion per tile, a
// CTA whose slice held many short portions ran partial tiles at the pace of
// full ones and finished last.
//
// Data movement. Each (block, kv head) of K and of V is a contiguous 16 x 128
// bf16 tile in the cache. Tiled TMA sees the cache as a 4-D tensor {64 dims,
// 8 rows, 2 halves, 8-row groups} (strides 256 B, 128 B, 2 KB), so ONE 4 KB
// copy lands a block already in the 128B-swizzled layout the MMAs read (8-key
// groups 2 KB apart, the two 64-dim halves of a group 1 KB apart): at this
// rate of copies per SM, the count of copies, not their bytes, would set the
// pace with 2 KB copies. Eight blocks per stage, three stages of 68 KB (K, V
// and the q rows of the tile's portions). Block ids are loaded two tiles
// ahead of their use.
//
// Warp roles (192 threads, one CTA per SM): warps 0-3 softmax and epilogue
// (warp w reads TMEM lanes 32w .. 32w+31), warp 4 the TMA producer (it also
// walks the work list and publishes a record per tile), warp 5 allocates TMEM
// and one of its threads issues the MMAs: each tile's S as soon as the tile
// has landed (so the next S is ready while the softmax of the current tile
// runs), each tile's P.V as soon as its softmax is done. Every wait is
// bounded; one that gives up sets the device error word and the CTA winds
// down.
#include <cuda.h>
#include <cuda_bf16.h>

#include <type_traits>

#include "pa_internal.h"
#include "ptx.cuh"

namespace pa {

namespace {

constexpr unsigned kAllLanes = 0xffffffffu;
constexpr int kD = 128;                   // head dim of this kernel
constexpr int kStages = 3;
constexpr int kTileBlocks = 8;            // 16-key cache blocks per 128-key tile
// A K or V tile (128 keys x 128 dims) in shared memory: 16 groups of 8 keys,
// 2 KB apart; in a group, the 64-dim half h 1 KB in, as 8 rows of 128 B
// (128B-swizzled). One TMA copy lands a 16-key block: 2 groups x 2 halves.
constexpr int kGroup = 2048;              // stride of 8-key groups
constexpr int kHalfOff = 1024;            // offset of the second 64-dim half in a group
constexpr int kKvTile = 16 * kGroup;      // K (or V) of one tile: 32 KB
constexpr int kNhalf = 16 * 128;          // one half of a 16-row N operand (q rows, P^T)
constexpr int kNbuf = 2 * kNhalf;
constexpr int kWarps = 6;
constexpr int kThreads = 32 * kWarps;
constexpr int kTmemCols = 64;             // S (2 x 16 columns), O (16 columns)
constexpr uint32_t kTmS = 0, kTmO = 32;

// Shared memory, from a 1024-byte aligned base. A stage holds one 128-key
// tile: K, V, and the q rows of the (at most two) portions it covers.
constexpr int kQBytes = 2 * kNhalf;            // q rows: [2 slots][2 halves][8 rows][128 B]
constexpr int kStageBytes = 2 * kKvTile + kQBytes;
constexpr int OFF_STAGE = 0;
constexpr int OFF_P = kStages * kStageBytes;   // 2 buffers of P^T
constexpr int OFF_REC = OFF_P + 2 * kNbuf;     // one tile record per stage
constexpr int OFF_XCH = OFF_REC + kStages * 64;  // [2][4 warps][16] floats
enum : int {
  B_FULL = 0 /* x3 */, B_EMPTY = 3 /* x3 */, B_S = 6 /* x2 */, B_PREADY = 8 /* x2 */,
  B_PFREE = 10 /* x2 */, B_XCH = 12 /* x2 */, B_DRAIN = 14, B_COUNT = 15
};
constexpr int OFF_BAR = OFF_XCH + 2 * 4 * 16 * 4;
constexpr int OFF_TSLOT = OFF_BAR + 8 * B_COUNT;
constexpr int OFF_UNITS = (OFF_TSLOT + 16 + 15) / 16 * 16;  // self-planned unit table
constexpr int kSmem = OFF_UNITS + (int)sizeof(UnitInfo) * (kSelfPlanMaxReqs + 1) + 1024;
static_assert(kSmem <= 227 * 1024, "one CTA per SM");

// A tile covers the end of one portion (a (token, kv head) part of this
// CTA's slice) and possibly the start of the next. Portion n of the CTA takes
// slot n % 2: its q rows are rows 8 * slot .. of the N operand, its scores
// and outputs columns 8 * slot .. of S^T and O^T.
constexpr int F_FIRST = 1;  // the portion's first tile
constexpr int F_LAST = 2;   // the portion's last tile
constexpr int F_WHOLE = 4;  // the portion is the whole (token, kv head): store bf16 output
constexpr int F_ACTIVE = 8; // the slot has rows in this tile
struct SlotRec {
  int tok, kv, key0, len, row0, nrows, flags, pad;  // rows row0 .. row0 + nrows - 1 hold keys key0 ..
};
struct Rec {
  SlotRec s[2];  // s[0].pad: 1 = no more tiles
};
static_assert(sizeof(Rec) == 64, "records are 64 bytes");

// Instruction descriptor, kind::f16 with bf16 A/B and fp32 D; a_mn / b_mn
// select the M/N-major (transposed) form of each operand.
constexpr uint32_t idesc_tc(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) |
         ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// TMEM loads/stores of N consecutive 32-bit columns of the warp's 32 lanes.
template <int N>
__device__ __forceinline__ void tm_ld(uint32_t taddr, uint32_t (&r)[N]) {
  if constexpr (N == 1) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(r[0]) : "r"(taddr) : "memory");
  } else if constexpr (N == 2) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x2.b32 {%0, %1}, [%2];"
                 : "=r"(r[0]), "=r"(r[1]) : "r"(taddr) : "memory");
  } else if constexpr (N == 4) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(taddr) : "memory");
  } else {
    static_assert(N == 8, "1, 2, 4 or 8 columns");
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr)
                 : "memory");
  }
}
template <int N>
__device__ __forceinline__ void tm_st(uint32_t taddr, const uint32_t (&r)[N]) {
  if constexpr (N == 1) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(r[0]) : "memory");
  } else if constexpr (N == 2) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x2.b32 [%0], {%1, %2};" ::"r"(taddr), "r"(r[0]),
                 "r"(r[1])
                 : "memory");
  } else if constexpr (N == 4) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3])
                 : "memory");
  } else {
    static_assert(N == 8, "1, 2, 4 or 8 columns");
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(
                     taddr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
  }
}

__device__ __forceinline__ uint16_t bf16_bits(float x) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

// After the transposing reduction below, the head whose value a lane holds.
template <int G>
__device__ __forceinline__ int tc_head_of_lane(int lane) {
  int h = 0;
#pragma unroll
  for (int st = 0; (1 << st) < G; ++st) h += ((lane >> st) & 1) * (G >> (st + 1));
  return h;
}

// Reduce G per-lane values over the 32 lanes of the warp, one result per head
// (max or sum). The first log2(G) rounds halve the live values (a lane keeps
// one half and sends its partner the other), the rest are plain butterflies;
// every lane ends with the warp's result for head tc_head_of_lane<G>(lane).
template <int G, bool MAX>
__device__ __forceinline__ float warp_reduce_heads(float (&v)[G], int lane) {
#pragma unroll
  for (int st = 0; st < 5; ++st) {
    const int m = 1 << st;
    const int n = (G >> st) > 1 ? (G >> st) : 1;
    if (n > 1) {
      const bool upper = (lane & m) != 0;
#pragma unroll
      for (int i = 0; i < n / 2; ++i) {
        const float send = upper ? v[i] : v[i + n / 2];
        const float keep = upper ? v[i + n / 2] : v[i];
        const float got = __shfl_xor_sync(kAllLanes, send, m);
        v[i] = MAX ? fmaxf(keep, got) : keep + got;
      }
    } else {
      const float got = __shfl_xor_sync(kAllLanes, v[0], m);
      v[0] = MAX ? fmaxf(v[0], got) : v[0] + got;
    }
  }
  return v[0];
}

}  // namespace

struct TcDecodeParams {
  CUtensorMap tm_q;  // q as {64, T * Hq rows, 2 halves}, box {64, 8, 2}, 128B swizzle
  CUtensorMap tm_k;  // k_cache as {64, 8, 2, blocks * Hkv * 2 groups}, box {64, 8, 2, 2}
  CUtensorMap tm_v;
  DecodeParams d;
};

template <int G>
__global__ void __launch_bounds__(kThreads, 1)
    pa_decode_tc_kernel(const __grid_constant__ TcDecodeParams tp) {
  const DecodeParams& p = tp.d;
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;  // swizzled operand tiles need 1024-byte alignment
  unsigned char* const gb = smem_raw + (base - raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // The merge pass may be placed as CTAs of this grid retire (it waits for
  // the whole grid before reading).
  griddep_launch_dependents();
  auto BAR = [&](int i) -> uint32_t { return base + OFF_BAR + 8u * (uint32_t)i; };
  auto wait = [&](int i, int parity) -> bool {
    if (mbar_wait_bounded(BAR(i), (uint32_t)parity & 1u)) return true;
    report_error(p.err, PA_DEVERR_WAIT_TIMEOUT, 2000 + i);
    return false;
  };
  Rec* const recs = reinterpret_cast<Rec*>(gb + OFF_REC);

  if (threadIdx.x == 0) {
    for (int i = 0; i < B_COUNT; ++i) {
      // P_READY and the exchanges are arrived at by the 128 softmax threads;
      // every other barrier once (an expect_tx arrive or an MMA commit).
      const bool by_softmax = i == B_PREADY || i == B_PREADY + 1 || i == B_XCH || i == B_XCH + 1;
      mbar_init(BAR(i), by_softmax ? 128 : 1);
    }
    fence_barrier_init();
  }
  // Rows past the group in each slot of the q and P^T operands stay zero for
  // good (TMA and the softmax write only the first G rows of a slot), and so
  // do the padded MMA columns.
  for (int st = 0; st < kStages; ++st)
    for (int idx = threadIdx.x; idx < kQBytes / 16; idx += kThreads)
      reinterpret_cast<uint4*>(gb + OFF_STAGE + st * kStageBytes + 2 * kKvTile)[idx] =
          make_uint4(0u, 0u, 0u, 0u);
  for (int idx = threadIdx.x; idx < (2 * kNbuf) / 16; idx += kThreads)
    reinterpret_cast<uint4*>(gb + OFF_P)[idx] = make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async_smem();
  if (warp == 5) {
    tmem_alloc(base + OFF_TSLOT, kTmemCols);
    tmem_relinquish();
  }

  // The work list: from the planner (the preceding grid), or - for a
  // decode-only batch - built here from query_start_loc and seq_lens without
  // waiting for any earlier grid. A unit without keys keeps len 0.
  const UnitInfo* units = p.units;
  int W, K;
  bool waited = false;  // griddepcontrol.wait done (the plan and the KV write are visible)
  if (p.self_plan) {
    UnitInfo* const su = reinterpret_cast<UnitInfo*>(gb + OFF_UNITS);
    __shared__ int s_tot[kWarps];
    const int R = p.num_reqs, T = p.num_tokens, Hkv_ = p.num_kv_heads;
    int carry = 0;
    for (int r0 = 0; r0 < R; r0 += kThreads) {
      const int r = r0 + (int)threadIdx.x;
      int n = 0, q0 = T, L = 0;
      if (r < R) {
        q0 = __ldg(p.qsl + r);
        const int q1 = __ldg(p.qsl + r + 1);
        L = __ldg(p.seq_lens + r);
        const int qlen = q1 - q0;
        if (q0 < 0 || q1 < q0 || q1 > T) {
          report_error(p.err, PA_DEVERR_QSL, r);
          q0 = T;
        } else if (L < qlen || qlen > 1 || (L + kBlockSize - 1) / kBlockSize > p.max_blocks_per_req ||
                   qlen > p.max_query_len || L > p.max_seq_len) {
          report_error(p.err, PA_DEVERR_LENGTHS, r);
        } else if (qlen == 1) {
          n = Hkv_ * ((L + kBlockSize - 1) / kBlockSize);
        }
      }
      int incl = n;  // warp inclusive scan of positions
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(kAllLanes, incl, o);
        if (lane >= o) incl += y;
      }
      if (lane == 31) s_tot[warp] = incl;
      __syncthreads();
      int off = carry;
      for (int w2 = 0; w2 < warp; ++w2) off += s_tot[w2];
      if (r < R) su[r] = UnitInfo{q0, r, n > 0 ? L : 0, off + incl - n};
      for (int w2 = 0; w2 < kWarps; ++w2) carry += s_tot[w2];
      __syncthreads();
    }
    if (threadIdx.x == 0) su[R] = UnitInfo{T, -1, 0, carry};
    if (blockIdx.x == 0 && threadIdx.x == 0) {  // the merge pass slices alike
      p.header_out->num_units = R;
      p.header_out->num_positions = carry;
    }
    units = su;
    W = carry;
    K = R;
  } else {
    griddep_wait();  // the plan is written by the preceding grid
    waited = true;
    W = p.header->num_positions;
    K = p.header->num_units;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(gb + OFF_TSLOT);

  const int Hkv = p.num_kv_heads, Hq = p.num_q_heads;
  const int w = (int)blockIdx.x;
  const int all = (int)gridDim.x < p.max_workers ? (int)gridDim.x : p.max_workers;
  const int NW = W > 0 ? plan_workers(W, all) : 0;
  int S = 0, E = 0;
  if (w < NW) {
    S = worker_begin(w, W, NW);
    E = worker_begin(w + 1, W, NW);
  }

  if (warp == 4) {
    // ======================= work walk + TMA producer =======================
    auto load_unit = [&](int k) -> UnitInfo {
      const int4 u = *reinterpret_cast<const int4*>(units + k);
      return UnitInfo{u.x, u.y, u.z, u.w};
    };
    // the walk: the portion holding position y is (unit k, kv head kv), at
    // block blk of its nb blocks; portion number np, first block pstart
    int k = 0;
    UnitInfo U{0, 0, 0, 0}, Un{0, 0, 0, 0};
    int nb = 1, kv = 0, blk = 0, y = S, pstart = 0, np = 0;
    bool pfirst = true;  // the current portion has not been in a tile yet
    if (S < E) {
      int lo = 0, hi = K;  // base[lo] <= S < base[hi]
      if (p.worker_unit && !p.self_plan) {
        lo = __ldg(p.worker_unit + w);
        hi = lo + 1;
      }
#pragma unroll 1
      while (hi - lo > 1) {
        const int step = (hi - lo + 31) / 32;
        const int idx = lo + lane * step;
        const bool ok = idx < hi && units[idx].base <= S;
        const unsigned bal = __ballot_sync(kAllLanes, ok);
        lo = lo + (31 - __clz(bal)) * step;
        hi = min(hi, lo + step);
      }
      k = lo;
      U = load_unit(k);
      Un = load_unit(k + 1);
      nb = (U.len + kBlockSize - 1) / kBlockSize;
      const int off = S - U.base;
      kv = off / nb;
      blk = off - kv * nb;
      pstart = blk;
      if (w > 0 && lane == 0) {  // the merge task of the slice boundary before this worker
        int4 task = make_int4(-1, 0, 0, 0);
        if (blk != 0) {
          const int first = S - blk;
          const int wf = worker_of(first, W, NW);
          if (w == wf + 1) task = make_int4(U.tok, kv, wf, worker_of(first + nb - 1, W, NW));
        }
        p.merge_tasks[w] = task;
      }
    }

    struct Meta {
      SlotRec s[2];
      int nblk;  // blocks in the tile; 0: no more tiles
      int last_blk;  // the tile holds a portion's last block (a decode's newest token)
      int pid, kvl;  // this lane's block id (loaded now, used two tiles later) and kv head
    };
    // The next tile: up to eight consecutive positions of the slice, from at
    // most two portions.
    auto next_tile = [&]() -> Meta {
      Meta t;
      t.nblk = 0;
      t.last_blk = 0;
      t.pid = 0;
      t.kvl = 0;
#pragma unroll
      for (int j = 0; j < 2; ++j) t.s[j] = SlotRec{0, 0, 0, 0, 0, 0, 0, 0};
      int used = 0;  // portions placed
      while (y < E && t.nblk < kTileBlocks && used < 2) {
        const int n = min(kTileBlocks - t.nblk, min(nb - blk, E - y));
        const int j = np & 1;
        const bool seg_done = blk + n == nb;
        const bool last = seg_done || y + n == E;
        const SlotRec sr{U.tok, kv, blk * kBlockSize, U.len, t.nblk * kBlockSize, n * kBlockSize,
                         F_ACTIVE | (pfirst ? F_FIRST : 0) | (last ? F_LAST : 0) |
                             ((last && seg_done && pstart == 0) ? F_WHOLE : 0),
                         0};
        if (j == 0) t.s[0] = sr; else t.s[1] = sr;
        if (seg_done) t.last_blk = 1;
        if (lane >= t.nblk && lane < t.nblk + n) {
          t.pid = __ldg(p.block_tables + (size_t)U.req * p.bt_stride + blk + (lane - t.nblk));
          t.kvl = kv;
        }
        pfirst = false;
        t.nblk += n;
        y += n;
        blk += n;
        ++used;
        if (blk == nb && y < E) {  // on to the next (token, kv head): a new portion
          blk = 0;
          pstart = 0;
          pfirst = true;
          ++np;
          if (++kv == Hkv) {
            kv = 0;
            // next unit with keys (units without any keep len 0)
            do {
              ++k;
              U = Un;
              Un = load_unit(k + 1);
            } while (U.len <= 0);
            nb = (U.len + kBlockSize - 1) / kBlockSize;
          }
        }
      }
      return t;
    };

    int i = 0;
    bool ok = true;
    // Issue one tile (cur) after computing the tile two ahead into nxt2; the
    // loop below rotates three descriptors at compile time instead of
    // copying them every tile (the producer's instructions are on the
    // critical path of a stage's turnaround).
    auto issue = [&](const Meta& cur, Meta& nxt2) -> bool {  // false: stop
      nxt2 = next_tile();
      const int st = i % kStages;
      if (i >= kStages && !wait(B_EMPTY + st, (i / kStages) - 1)) {
        ok = false;
        return false;
      }
      const uint32_t full = BAR(B_FULL + st);
      if (cur.nblk == 0) {
        if (lane == 0) {
          recs[st].s[0] = SlotRec{0, 0, 0, 0, 0, 0, 0, 1};
          recs[st].s[1] = SlotRec{0, 0, 0, 0, 0, 0, 0, 0};
          mbar_arrive(full);
        }
        ++i;
        return false;
      }
      const int nq = ((cur.s[0].flags & F_ACTIVE) ? 1 : 0) + ((cur.s[1].flags & F_ACTIVE) ? 1 : 0);
      if (lane == 0) {
        recs[st].s[0] = cur.s[0];
        recs[st].s[1] = cur.s[1];
        mbar_arrive_expect_tx(full, (uint32_t)cur.nblk * 2u * 4096u + (uint32_t)nq * 2048u);
      }
      __syncwarp();
      // a decode's newest token, written by the preceding grid, sits in its
      // last block: see that grid's writes before copying such a block
      if (!waited && cur.last_blk) {
        griddep_wait();
        waited = true;
      }
      const uint32_t sbase = base + OFF_STAGE + st * kStageBytes;
      if (lane < cur.nblk) {
        int pid = cur.pid;
        if (pid < 0 || pid >= p.num_blocks) {
          report_error(p.err, PA_DEVERR_BLOCK_ID, lane);
          pid = 0;
        }
        const int grp = (pid * Hkv + cur.kvl) * (kBlockSize / 8);  // the block's first 8-key group
        const uint32_t dst = sbase + lane * 2 * kGroup;
        tma_load_4d(dst, &tp.tm_k, 0, 0, 0, grp, full);
        tma_load_4d(dst + kKvTile, &tp.tm_v, 0, 0, 0, grp, full);
      }
      const int qflags = lane == 0 ? cur.s[0].flags : cur.s[1].flags;
      if (lane < 2 && (qflags & F_ACTIVE)) {  // q rows of slot `lane`
        const int qrow = lane == 0 ? cur.s[0].tok * Hq + cur.s[0].kv * G
                                   : cur.s[1].tok * Hq + cur.s[1].kv * G;
        // 8 q rows from the group's first (rows past the group are other
        // heads' queries, or zeros past the end: they only feed the slot's
        // unused columns)
        tma_load_3d(sbase + 2 * kKvTile + lane * kGroup, &tp.tm_q, 0, qrow, 0, full);
      }
      ++i;
      return true;
    };
    Meta ma = next_tile();
    Meta mb = next_tile();
    Meta mc;
#pragma unroll 1
    while (issue(ma, mc) && issue(mb, ma) && issue(mc, mb)) {
    }
    // every copy issued has landed before the CTA may exit
    for (int j = i > kStages ? i - kStages : 0; j < i; ++j)
      mbar_wait_bounded(BAR(B_FULL + j % kStages), (uint32_t)(j / kStages) & 1u);
  } else if (warp == 5) {
    // ======================= MMA issuer (lane 0) =======================
    // Two kinds of work, each in tile order: S(j) once tile j has landed and
    // S buffer j % 2 is free (the P.V of tile j - 2 issued, hence its softmax
    // done), and O(j) = P.V once the softmax of tile j is done. Whichever is
    // ready is issued, the P.V first: it frees a stage for the producer. O^T
    // always accumulates: its columns start at zero and an epilogue zeroes a
    // slot's columns after reading them.
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_tc(128, 16, false, false);
      constexpr uint32_t id_o = idesc_tc(128, 16, true, false);
      const uint64_t kdesc = smem_desc_sw128(base, 16, kGroup);         // K-major: K tile, q rows
      const uint64_t pdesc = smem_desc_sw128(base, 16, 1024);           // K-major: P^T
      const uint64_t vdesc = smem_desc_sw128(base, kHalfOff, kGroup);   // M/N-major: V^T
      int ns = 0, no = 0;  // next tile for S, next tile for P.V
      bool end_seen = false;
      uint32_t spins = 0;
      uint64_t t0 = 0;
#pragma unroll 1
      while (!(end_seen && no == ns)) {
        if (no < ns && mbar_test(BAR(B_PREADY + (no & 1)), (uint32_t)(no >> 1) & 1u)) {
          tc_fence_after();
          const int st = no % kStages;
          const uint64_t a0 = vdesc + ((uint64_t)(OFF_STAGE + st * kStageBytes + kKvTile) >> 4);
          const uint64_t b0 = pdesc + ((uint64_t)(OFF_P + (no & 1) * kNbuf) >> 4);
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)  // keys 16 ks .. 16 ks + 15: groups 2 ks, 2 ks + 1
            umma_bf16(tmem + kTmO, a0 + (uint64_t)((ks * 2 * kGroup) >> 4),
                      b0 + (uint64_t)(((ks >> 2) * kNhalf + (ks & 3) * 32) >> 4), id_o, 1u);
          umma_commit(BAR(B_EMPTY + st));
          umma_commit(BAR(B_PFREE + (no & 1)));
          ++no;
          spins = 0;
        } else if (!end_seen && ns <= no + 1 &&
                   mbar_test(BAR(B_FULL + ns % kStages), (uint32_t)(ns / kStages) & 1u)) {
          const int st = ns % kStages;
          if (recs[st].s[0].pad) {
            end_seen = true;
          } else {
            tc_fence_after();
            const uint64_t a0 = kdesc + ((uint64_t)(OFF_STAGE + st * kStageBytes) >> 4);
            const uint64_t b0 = kdesc + ((uint64_t)(OFF_STAGE + st * kStageBytes + 2 * kKvTile) >> 4);
#pragma unroll
            for (int ks = 0; ks < kD / 16; ++ks)  // head dims 16 ks .. 16 ks + 15
              umma_bf16(tmem + kTmS + 16 * (ns & 1),
                        a0 + (uint64_t)(((ks >> 2) * kHalfOff + (ks & 3) * 32) >> 4),
                        b0 + (uint64_t)(((ks >> 2) * kHalfOff + (ks & 3) * 32) >> 4), id_s,
                        ks > 0 ? 1u : 0u);
            umma_commit(BAR(B_S + (ns & 1)));
            ++ns;
          }
          spins = 0;
        } else if (++spins > 64) {  // nothing ready: give up after ~2 s without progress
          if (spins == 65) t0 = global_timer_ns();
          if (global_timer_ns() - t0 > 2000000000ull) {
            report_error(p.err, PA_DEVERR_WAIT_TIMEOUT, 2000 + B_PREADY);
            break;
          }
        }
      }
      // every MMA issued above has completed before TMEM is released
      umma_commit(BAR(B_DRAIN));
      mbar_wait_bounded(BAR(B_DRAIN), 0);
    }
    __syncwarp();
  } else {
    // ======================= softmax + epilogue (warps 0-3) =======================
    const int m = warp * 32 + lane;  // key row of S^T and head dim of O^T: the TMEM lane
    const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
    float* const xch = reinterpret_cast<float*>(gb + OFF_XCH);
    int nx = 0;  // exchanges done
    // Per-(slot, head) max or sum over the 128 softmax threads: warp
    // reduction, then the four warps meet on an mbarrier (bounded wait).
    // Exchange k uses buffer and barrier k % 2: a buffer is rewritten only
    // after every thread has passed the other barrier, i.e. has read this one.
    auto block_reduce = [&](auto& v, auto tag_n, bool is_max) -> bool {
      constexpr int N = decltype(tag_n)::value;
      const float x = is_max ? warp_reduce_heads<N, true>(v, lane) : warp_reduce_heads<N, false>(v, lane);
      const int kx = nx++;
      float* const xb = xch + (kx & 1) * 64;
      if (lane < N) xb[warp * 16 + tc_head_of_lane<N>(lane)] = x;
      mbar_arrive(BAR(B_XCH + (kx & 1)));
      if (!wait(B_XCH + (kx & 1), kx >> 1)) return false;
#pragma unroll
      for (int h = 0; h < N; ++h) {
        const float a = xb[h], b = xb[16 + h], c = xb[32 + h], d = xb[48 + h];
        v[h] = is_max ? fmaxf(fmaxf(a, b), fmaxf(c, d)) : (a + b) + (c + d);
      }
      return true;
    };
    // O^T starts at zero (the P.V MMAs always accumulate)
    {
      uint32_t z[16];
#pragma unroll
      for (int c = 0; c < 16; ++c) z[c] = 0u;
      tm_st<8>(trow + kTmO, *reinterpret_cast<uint32_t(*)[8]>(z));
      tm_st<8>(trow + kTmO + 8, *reinterpret_cast<uint32_t(*)[8]>(z + 8));
      tmem_wait_st();
    }
    float mref[2][G], lth[2][G];
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int h = 0; h < G; ++h) {
        mref[j][h] = 0.f;
        lth[j][h] = 0.f;
      }
    // P^T rows of slot j in buffer b may be non-zero: bit 2b + j (uniform)
    int dirty = 0;
    // P^T[8 slot + h][m] of buffer b: row 8 slot + h, 16-byte unit (m % 64) / 8
    // swizzled by h, half m / 64
    auto prow = [&](int b, int j, int h) -> uint16_t* {
      return reinterpret_cast<uint16_t*>(gb + OFF_P + b * kNbuf + (m >> 6) * kNhalf + j * 1024 +
                                         h * 128 + ((((m & 63) >> 3) ^ h) << 4) + (m & 7) * 2);
    };
    int i = 0;
    bool ok = true;
#pragma unroll 1
    while (ok) {
      const int st = i % kStages;
      if (!wait(B_FULL + st, i / kStages)) { ok = false; break; }  // the tile record is visible
      const SlotRec r0 = recs[st].s[0], r1 = recs[st].s[1];
      if (r0.pad) break;
      if (!wait(B_S + (i & 1), i >> 1)) { ok = false; break; }
      tc_fence_after();
      const int b = i & 1;
      // this thread's key: slot my (-1: no key), valid when inside its sequence
      const bool in0 = (r0.flags & F_ACTIVE) && m >= r0.row0 && m < r0.row0 + r0.nrows;
      const bool in1 = (r1.flags & F_ACTIVE) && m >= r1.row0 && m < r1.row0 + r1.nrows;
      const int my = in0 ? 0 : (in1 ? 1 : -1);
      const bool valid = in0 ? (r0.key0 + (m - r0.row0) < r0.len)
                             : (in1 ? (r1.key0 + (m - r1.row0) < r1.len) : false);
      // P^T buffer b is free once the P.V of tile i - 2 has completed
      if (i >= 2 && !wait(B_PFREE + b, (i - 2) >> 1)) { ok = false; break; }
      // One pass per active slot (two only where the tile crosses from one
      // portion into the next): the slot's scores, its maxima, P^T rows.
      const int nact = ((r0.flags & F_ACTIVE) ? 1 : 0) + ((r1.flags & F_ACTIVE) ? 1 : 0);
#pragma unroll 1
      for (int pass = 0; pass < nact; ++pass) {
        const int jj = (pass == 0 && (r0.flags & F_ACTIVE)) ? 0 : 1;
        const int fl = jj ? r1.flags : r0.flags;
        const bool mine = valid && my == jj;  // this thread's key belongs to slot jj
        uint32_t sr[G];
        tm_ld<G>(trow + kTmS + 16 * b + 8 * jj, sr);
        tmem_wait_ld();
        float t[G], tm[G], mr[G], lt[G];
#pragma unroll
        for (int h = 0; h < G; ++h) {
          t[h] = mine ? __uint_as_float(sr[h]) * p.scale_log2 : -INFINITY;
          tm[h] = t[h];
          mr[h] = jj ? mref[1][h] : mref[0][h];
          lt[h] = jj ? lth[1][h] : lth[0][h];
        }
        if (!block_reduce(tm, std::integral_constant<int, G>{}, true)) { ok = false; break; }
        // reference maxima: a portion's first tile sets them (it holds the
        // portion's first key, so they are finite); later tiles move them
        // only by more than 2^8, rescaling the slot's O^T columns
        bool resc = false;
        float alpha[G];
#pragma unroll
        for (int h = 0; h < G; ++h) {
          alpha[h] = 1.f;
          if (fl & F_FIRST) {
            mr[h] = tm[h];
            lt[h] = 0.f;
          } else if (tm[h] > mr[h] + 8.f) {
            alpha[h] = exp2f(mr[h] - tm[h]);
            mr[h] = tm[h];
            resc = true;
          }
        }
        if (resc) {  // uniform: every thread holds the same maxima
          // O^T is stable once the previous tile's P.V has completed
          if (!wait(B_PFREE + ((i - 1) & 1), (i - 1) >> 1)) { ok = false; break; }
          tc_fence_after();
          uint32_t o[G];
          tm_ld<G>(trow + kTmO + 8 * jj, o);
          tmem_wait_ld();
#pragma unroll
          for (int h = 0; h < G; ++h) {
            o[h] = __float_as_uint(__uint_as_float(o[h]) * alpha[h]);
            lt[h] *= alpha[h];
          }
          tm_st<G>(trow + kTmO + 8 * jj, o);
          tmem_wait_st();
        }
        float pr[G];
#pragma unroll
        for (int h = 0; h < G; ++h) {
          pr[h] = mine ? ex2_approx(t[h] - mr[h]) : 0.f;
          lt[h] += pr[h];
        }
#pragma unroll
        for (int h = 0; h < G; ++h) {
          if (jj) {
            mref[1][h] = mr[h];
            lth[1][h] = lt[h];
          } else {
            mref[0][h] = mr[h];
            lth[0][h] = lt[h];
          }
        }
#pragma unroll
        for (int h = 0; h < G; ++h) *prow(b, jj, h) = bf16_bits(pr[h]);
        dirty |= 1 << (2 * b + jj);
        if (nact == 1 && (dirty & (1 << (2 * b + (1 - jj))))) {  // the idle slot's rows to zero
#pragma unroll
          for (int h = 0; h < G; ++h) *prow(b, 1 - jj, h) = 0;
          dirty &= ~(1 << (2 * b + (1 - jj)));
        }
      }
      if (!ok) break;
      if (!valid) {
        // A key past the sequence end (or a block slot this tile did not
        // load) has P = 0, but its V row may hold anything, NaN included, and
        // 0 * NaN would poison O: clear the row.
        unsigned char* const vrow =
            gb + OFF_STAGE + st * kStageBytes + kKvTile + (m >> 3) * kGroup + (m & 7) * 128;
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int q = 0; q < 8; ++q)
            *reinterpret_cast<uint4*>(vrow + c * kHalfOff + q * 16) = make_uint4(0u, 0u, 0u, 0u);
      }
      fence_proxy_async_smem();  // generic-proxy stores -> visible to the tensor core
      tc_fence_before();
      mbar_arrive(BAR(B_PREADY + (i & 1)));

      if ((r0.flags | r1.flags) & F_LAST) {
        // ---- epilogue of the portions ending here: O^T complete once tile
        // i's P.V is ----
        if (!wait(B_PFREE + (i & 1), i >> 1)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const SlotRec rc = j == 0 ? r0 : r1;
          if (!(rc.flags & F_LAST)) continue;
          float ls[G];
#pragma unroll
          for (int h = 0; h < G; ++h) ls[h] = lth[j][h];
          if (!block_reduce(ls, std::integral_constant<int, G>{}, false)) { ok = false; break; }
          uint32_t o[8];
          tm_ld<8>(trow + kTmO + 8 * j, o);
          tmem_wait_ld();
          if (rc.flags & F_WHOLE) {
            uint16_t* const orow = p.out + ((size_t)rc.tok * Hq + (size_t)rc.kv * G) * kD + m;
#pragma unroll
            for (int h = 0; h < G; ++h)
              orow[h * kD] = bf16_bits(__uint_as_float(o[h]) * (p.v_scale / ls[h]));
          } else {
            // a partial (m, l, o) for the merge pass in slot u + w: tokens
            // increase with the position order, so the slot is unique per portion
            float* const slot =
                p.partials + (size_t)(rc.tok * Hkv + rc.kv + w) * (size_t)p.slot_floats;
            if (m == 0) {
#pragma unroll
              for (int h = 0; h < G; ++h) {
                __stcg(slot + h, mref[j][h]);
                __stcg(slot + G + h, ls[h]);
              }
            }
#pragma unroll
            for (int h = 0; h < G; ++h) __stcg(slot + 16 + h * kD + m, __uint_as_float(o[h]));
          }
          // the slot's columns start the next portion at zero
          uint32_t z[8];
#pragma unroll
          for (int c = 0; c < 8; ++c) z[c] = 0u;
          tm_st<8>(trow + kTmO + 8 * j, z);
          tmem_wait_st();
        }
        if (!ok) break;
        tc_fence_before();  // the next tile's P.V accumulates into O^T
      }
      ++i;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------------------
namespace {

template <int G>
cudaError_t launch_tc_t(const DecodeParams& d, int grid, cudaStream_t s) {
  TcDecodeParams tp;
  tp.d = d;
  // q as {64 dims, rows, 2 halves}: a box of 8 rows lands as [half][8 rows][128 B]
  const uint64_t qrows = (uint64_t)d.num_tokens * (uint64_t)d.num_q_heads;
  const uint64_t qd[3] = {64, qrows, 2}, qs[2] = {kD * 2, 128};
  const uint32_t qb[3] = {64, 8, 2};
  // a cache as {64 dims, 8 rows, 2 halves, 8-row groups}: a box of 2 groups
  // (one 16-key block) lands as [group][half][8 rows][128 B]
  const uint64_t groups = (uint64_t)d.num_blocks * (uint64_t)d.num_kv_heads * (kBlockSize / 8);
  const uint64_t cd[4] = {64, 8, 2, groups}, cs[3] = {kD * 2, 128, 8 * kD * 2};
  const uint32_t cb[4] = {64, 8, 2, kBlockSize / 8};
  if (!encode_tmap_bf16(&tp.tm_q, 3, d.q, qd, qs, qb) ||
      !encode_tmap_bf16(&tp.tm_k, 4, d.k_cache, cd, cs, cb) ||
      !encode_tmap_bf16(&tp.tm_v, 4, d.v_cache, cd, cs, cb))
    return cudaErrorInvalidValue;
  auto kern = pa_decode_tc_kernel<G>;
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = s;
  // Programmatic launch: the grid starts when the preceding grid triggers
  // (the KV write at its top for a self-planned batch; otherwise the planner
  // or the tensor-core prefill grid, at their end).
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tp);
}

}  // namespace

int decode_tc_workers(int num_sms) {
  return num_sms < kMaxDecodeWorkers ? num_sms : kMaxDecodeWorkers;
}

bool decode_tc_supported(int head_dim, int group, bool f8, int key_start_blocks) {
  return head_dim == kD && !f8 && key_start_blocks == 0 &&
         (group == 1 || group == 2 || group == 4 || group == 8);
}

cudaError_t launch_decode_tc(const DecodeParams& p, int group, int num_sms, cudaStream_t s,
                             int* workers_out) {
  const int grid = decode_tc_workers(num_sms);
  *workers_out = grid;
  switch (group) {
    case 1: return launch_tc_t<1>(p, grid, s);
    case 2: return launch_tc_t<2>(p, grid, s);
    case 4: return launch_tc_t<4>(p, grid, s);
    case 8: return launch_tc_t<8>(p, grid, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace pa
