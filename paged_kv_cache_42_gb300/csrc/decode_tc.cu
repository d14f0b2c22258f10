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
//                    tile's max over 128 keys where needed (warp shuffles,
//                    then a 4-warp exchange on an mbarrier), exp2; P^T
//                    rounded to bf16 into shared memory in the B-operand
//                    layout.
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
// E4M3 caches (the F8 instantiation; "vLLM: An Exhaustive Technical Study for
// Kernel Engineers", 2.8: E4M3 codes with per-tensor k_scale / v_scale). Both
// products run as tcgen05.mma kind::f8f6f4 straight on the cached codes, so
// nothing widens K or V:
//   S^T = K Q'^T     each query row q is scaled by a power of two 2^e that
//                    brings its largest magnitude into [128, 256) and split
//                    into two E4M3 terms, q 2^e = hi + lo (exact for every
//                    element within 2^9 of the row's largest), by a small
//                    kernel before this one (launch_qsplit). N = 32: per slot,
//                    8 rows of hi then 8 of lo; the softmax adds the two
//                    column groups and undoes 2^e.
//   O^T += V^T P'^T  P' = 256 p against a reference max, set 1 above the
//                    maxima it comes from, that moves whenever a tile's max
//                    exceeds it by more than 0.75 (so P' <= 430, inside
//                    E4M3's 448), split the same way into hi + lo (a
//                    relative error near 2^-8, as bf16's); O^T keeps the two
//                    column groups apart until the epilogue.
// An E4M3 block is one 2 KB copy per tensor ([16 keys][128 B] rows are
// already the swizzle width), a stage 36 KB, five stages. A stage is sent a
// portion's q' rows only when it does not hold them already.
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
constexpr int kTileBlocks = 8;            // 16-key cache blocks per 128-key tile
constexpr int kWarps = 6;
constexpr int kThreads = 32 * kWarps;

// Shared-memory and TMEM layout of each instantiation, from a 1024-byte
// aligned base. A stage holds one 128-key tile: K, V, and the query operand
// rows of the (at most two) portions it covers.
template <bool F8>
struct TcL;
// bf16 cache. A K or V tile (128 keys x 128 dims): 16 groups of 8 keys, 2 KB
// apart; in a group, the 64-dim half h 1 KB in, as 8 rows of 128 B
// (128B-swizzled). One TMA copy lands a 16-key block: 2 groups x 2 halves.
// The q operand: [2 slots][2 halves][8 rows][128 B]; P^T: [2 key halves][16
// rows][128 B]. N = 16: slot s is rows / columns 8 s .. 8 s + 7.
template <>
struct TcL<false> {
  static constexpr int kStages = 3;
  static constexpr int kGroup = 2048;      // K operand: stride of 8-row groups (SBO)
  static constexpr int kHalfOff = 1024;    // second 64-dim half within a group
  static constexpr int kKvTile = 32768;
  static constexpr int kQBytes = 4096;
  static constexpr int kN = 16;            // MMA N, columns of S^T and O^T
  static constexpr int kSlotCols = 8;      // columns of one slot
  static constexpr int kKStep = 16;        // MMA K per instruction (elements)
  static constexpr int kPBytes = 4096;
  static constexpr uint32_t kTmemCols = 64;
};
// E4M3 cache. A K or V tile: [128 keys][128 B] (one 2 KB copy per block);
// the q' operand: [2 slots][hi, lo][8 rows][128 B] (1/2^e travels in the tile
// record); P'^T: [32 rows][128 B]. N = 32: slot s is rows / columns 16 s ..,
// the hi terms first.
template <>
struct TcL<true> {
  static constexpr int kStages = 5;
  static constexpr int kGroup = 1024;
  static constexpr int kHalfOff = 0;
  static constexpr int kKvTile = 16384;
  static constexpr int kQBytes = 4096;
  static constexpr int kN = 32;
  static constexpr int kSlotCols = 16;
  static constexpr int kKStep = 32;
  static constexpr int kPBytes = 4096;
  static constexpr uint32_t kTmemCols = 128;
};

// S^T in TMEM and P^T in shared memory are kept in this many buffers: a
// tile's S can be computed while the softmax of the tile before runs (three
// buffers measured no faster).
constexpr int kSP = 2;

template <bool F8>
struct TcSmem {
  using L = TcL<F8>;
  static constexpr int kStageBytes = 2 * L::kKvTile + L::kQBytes;
  static constexpr int OFF_STAGE = 0;
  static constexpr int OFF_P = L::kStages * kStageBytes;    // kSP buffers of P^T
  static constexpr int OFF_REC = OFF_P + kSP * L::kPBytes;  // one tile record per stage
  // E4M3: per stage, the inverse query scales of the tile's two slots ([2][8]
  // floats), and which portion's q' rows each stage holds per slot
  static constexpr int OFF_INV = OFF_REC + L::kStages * 64;
  static constexpr int OFF_QTAG = OFF_INV + L::kStages * 64;
  static constexpr int OFF_XCH = OFF_QTAG + 64;  // [2][4 warps][16] floats
  static constexpr int OFF_BAR = OFF_XCH + 2 * 4 * 16 * 4;
  // barriers: FULL[stages], EMPTY[stages], S[kSP], P_READY[kSP], P_FREE[kSP], XCH[2], DRAIN
  static constexpr int B_FULL = 0, B_EMPTY = L::kStages, B_S = 2 * L::kStages,
                       B_PREADY = B_S + kSP, B_PFREE = B_S + 2 * kSP, B_XCH = B_S + 3 * kSP,
                       B_DRAIN = B_XCH + 2, B_COUNT = B_DRAIN + 1;
  static constexpr int OFF_TSLOT = OFF_BAR + 8 * B_COUNT;
  static constexpr int OFF_UNITS = (OFF_TSLOT + 16 + 15) / 16 * 16;  // self-planned unit table
  static constexpr int SMEM = OFF_UNITS + (int)sizeof(UnitInfo) * (kSelfPlanMaxReqs + 1) + 1024;
  static_assert(SMEM <= 227 * 1024, "one CTA per SM");
  static_assert(kStageBytes % 1024 == 0, "stages keep the 1024-byte alignment of swizzled tiles");
  // TMEM columns: S^T buffers at 0, kN, 2 kN, O^T after them
  static constexpr uint32_t kTmS = 0, kTmO = kSP * L::kN;
  static_assert(kTmO + L::kN <= L::kTmemCols, "S^T buffers and O^T fit the allocation");
};

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
  // bf16: q as {64, T * Hq rows, 2 halves}, box {64, 8, 2}; a cache as
  // {64, 8, 2, blocks * Hkv * 2 groups}, box {64, 8, 2, 2}.
  // E4M3: the split q' rows as {128 B, T * Hq rows, 2 (hi, lo)}, box
  // {128, 8, 2}; a cache as {128 B, blocks * Hkv * 16 rows}, box {128, 16}.
  CUtensorMap tm_q;
  CUtensorMap tm_k;
  CUtensorMap tm_v;
  DecodeParams d;
};

template <int G, bool F8>
__global__ void __launch_bounds__(kThreads, 1)
    pa_decode_tc_kernel(const __grid_constant__ TcDecodeParams tp) {
  using L = TcL<F8>;
  using M = TcSmem<F8>;
  constexpr int kStages = L::kStages;
  const DecodeParams& p = tp.d;
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;  // swizzled operand tiles need 1024-byte alignment
  unsigned char* const gb = smem_raw + (base - raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // The merge pass may be placed as CTAs of this grid retire (it waits for
  // the whole grid before reading).
  griddep_launch_dependents();
  auto BAR = [&](int i) -> uint32_t { return base + M::OFF_BAR + 8u * (uint32_t)i; };
  auto wait = [&](int i, int parity) -> bool {
    if (mbar_wait_bounded(BAR(i), (uint32_t)parity & 1u)) return true;
    report_error(p.err, PA_DEVERR_WAIT_TIMEOUT, 2000 + i);
    return false;
  };
  Rec* const recs = reinterpret_cast<Rec*>(gb + M::OFF_REC);

  if (threadIdx.x == 0) {
    for (int i = 0; i < M::B_COUNT; ++i) {
      // P_READY and the exchanges are arrived at by the 128 softmax threads;
      // every other barrier once (an expect_tx arrive or an MMA commit).
      const bool by_softmax = (i >= M::B_PREADY && i < M::B_PREADY + kSP) || i == M::B_XCH ||
                              i == M::B_XCH + 1;
      mbar_init(BAR(i), by_softmax ? 128 : 1);
    }
    fence_barrier_init();
  }
  // The query operands of every stage and the P^T buffers start at zero:
  // rows past the group stay zero (bf16) or hold other heads' rows (TMA
  // copies 8 rows per slot), which only reach the slot's unused columns.
  for (int st = 0; st < kStages; ++st)
    for (int idx = threadIdx.x; idx < L::kQBytes / 16; idx += kThreads)
      reinterpret_cast<uint4*>(gb + M::OFF_STAGE + st * M::kStageBytes + 2 * L::kKvTile)[idx] =
          make_uint4(0u, 0u, 0u, 0u);
  for (int idx = threadIdx.x; idx < (kSP * L::kPBytes) / 16; idx += kThreads)
    reinterpret_cast<uint4*>(gb + M::OFF_P)[idx] = make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async_smem();
  if (warp == 5) {
    tmem_alloc(base + M::OFF_TSLOT, L::kTmemCols);
    tmem_relinquish();
  }

  // The work list: from the planner (the preceding grid), or - for a
  // decode-only batch - built here from query_start_loc and seq_lens without
  // waiting for any earlier grid. A unit without keys keeps len 0.
  const UnitInfo* units = p.units;
  int W, K;
  bool waited = false;  // griddepcontrol.wait done (the plan and the KV write are visible)
  if (p.self_plan) {
    UnitInfo* const su = reinterpret_cast<UnitInfo*>(gb + M::OFF_UNITS);
    __shared__ int s_tot[kWarps];
    const int R = p.num_reqs, T = p.num_tokens, Hkv_ = p.num_kv_heads;
    int carry = 0;
    for (int r0 = 0; r0 < R; r0 += kThreads) {
      const int r = r0 + (int)threadIdx.x;
      int n = 0, q0 = T, Lr = 0;
      if (r < R) {
        q0 = __ldg(p.qsl + r);
        const int q1 = __ldg(p.qsl + r + 1);
        Lr = __ldg(p.seq_lens + r);
        const int qlen = q1 - q0;
        if (q0 < 0 || q1 < q0 || q1 > T) {
          report_error(p.err, PA_DEVERR_QSL, r);
          q0 = T;
        } else if (Lr < qlen || qlen > 1 || (Lr + kBlockSize - 1) / kBlockSize > p.max_blocks_per_req ||
                   qlen > p.max_query_len || Lr > p.max_seq_len) {
          report_error(p.err, PA_DEVERR_LENGTHS, r);
        } else if (qlen == 1) {
          n = Hkv_ * ((Lr + kBlockSize - 1) / kBlockSize);
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
      if (r < R) su[r] = UnitInfo{q0, r, n > 0 ? Lr : 0, off + incl - n};
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
  } else if (p.overlap) {
    // started by the prefill-chunk grid once it had read the plan: the
    // planner and the KV write before it are complete; this grid waits for
    // the prefill-chunk grid only before it completes (see the end)
    waited = true;
    W = __ldcg(&p.header->num_positions);
    K = __ldcg(&p.header->num_units);
  } else {
    griddep_wait();  // the plan is written by the preceding grid
    waited = true;
    W = p.header->num_positions;
    K = p.header->num_units;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(gb + M::OFF_TSLOT);

  const int Hkv = p.num_kv_heads, Hq = p.num_q_heads;
  const int kstart = p.key_start_blocks;  // blocks of a cascade's common prefix, skipped here
  const int w = (int)blockIdx.x;
  int all = (int)gridDim.x < p.max_workers ? (int)gridDim.x : p.max_workers;
  if (p.overlap) all = min(all, __ldcg(&p.header->decode_workers));
  const int NW = W > 0 ? plan_workers(W, all) : 0;
  int S = 0, E = 0;
  if (w < NW) {
    S = worker_begin(w, W, NW);
    E = worker_begin(w + 1, W, NW);
  }

  if (warp == 4) {
    // ======================= work walk + TMA producer =======================
    // the planner's table (global memory, written by an earlier grid) is read
    // from L2; a self-planned one sits in shared memory
    auto load_unit = [&](int k) -> UnitInfo {
      const int4 u = p.self_plan ? *reinterpret_cast<const int4*>(units + k)
                                 : __ldcg(reinterpret_cast<const int4*>(units + k));
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
        lo = __ldcg(p.worker_unit + w);
        hi = lo + 1;
      }
#pragma unroll 1
      while (hi - lo > 1) {
        const int step = (hi - lo + 31) / 32;
        const int idx = lo + lane * step;
        const bool ok = idx < hi && load_unit(idx).base <= S;
        const unsigned bal = __ballot_sync(kAllLanes, ok);
        lo = lo + (31 - __clz(bal)) * step;
        hi = min(hi, lo + step);
      }
      k = lo;
      U = load_unit(k);
      Un = load_unit(k + 1);
      nb = max(1, (U.len + kBlockSize - 1) / kBlockSize - kstart);
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
    if constexpr (F8) {
      // the split query rows come from the preceding grid (launch_qsplit)
      if (!waited) {
        griddep_wait();
        waited = true;
      }
    }

    struct Meta {
      SlotRec s[2];
      int nblk;      // blocks in the tile; 0: no more tiles
      int last_blk;  // the tile holds a portion's last block (a decode's newest token)
      int pid, kvl;  // this lane's block id (loaded now, used two tiles later) and kv head
      float invl;    // E4M3: lanes 8 j + h hold slot j's inverse query scale of head h
    };
    // The next tile: up to eight consecutive positions of the slice, from at
    // most two portions.
    auto next_tile = [&]() -> Meta {
      Meta t;
      t.nblk = 0;
      t.last_blk = 0;
      t.pid = 0;
      t.kvl = 0;
      t.invl = 0.f;
#pragma unroll
      for (int j = 0; j < 2; ++j) t.s[j] = SlotRec{0, 0, 0, 0, 0, 0, 0, 0};
      int used = 0;  // portions placed
      while (y < E && t.nblk < kTileBlocks && used < 2) {
        const int n = min(kTileBlocks - t.nblk, min(nb - blk, E - y));
        const int j = np & 1;
        const bool seg_done = blk + n == nb;
        const bool last = seg_done || y + n == E;
        const SlotRec sr{U.tok, kv, (kstart + blk) * kBlockSize, U.len, t.nblk * kBlockSize,
                         n * kBlockSize,
                         F_ACTIVE | (pfirst ? F_FIRST : 0) | (last ? F_LAST : 0) |
                             ((last && seg_done && pstart == 0) ? F_WHOLE : 0),
                         0};
        if (j == 0) t.s[0] = sr; else t.s[1] = sr;
        if (seg_done) t.last_blk = 1;
        if (F8 && (lane >> 3) == j)
          t.invl = __ldg(p.qinv + ((size_t)U.tok * Hkv + kv) * 8 + (lane & 7));
        if (lane >= t.nblk && lane < t.nblk + n) {
          t.pid = __ldg(p.block_tables + (size_t)U.req * p.bt_stride + kstart + blk + (lane - t.nblk));
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
            nb = max(1, (U.len + kBlockSize - 1) / kBlockSize - kstart);
          }
        }
      }
      return t;
    };

    int i = 0;
    bool ok = true;
    int* const qtag = reinterpret_cast<int*>(gb + M::OFF_QTAG);
    if (F8) {
      if (lane < 2 * kStages) qtag[lane] = -1;
      __syncwarp();
    }
    // Issue one tile (cur) after computing the tile two ahead into nxt2; the
    // loop below rotates three descriptors at compile time instead of
    // copying them every tile (the producer's instructions are on the
    // critical path of a stage's turnaround).
    auto issue = [&](const Meta& cur, Meta& nxt2) -> bool {  // false: stop
      nxt2 = next_tile();
      const int st = i % kStages;
      if (i >= kStages && !wait(M::B_EMPTY + st, (i / kStages) - 1)) {
        ok = false;
        return false;
      }
      const uint32_t full = BAR(M::B_FULL + st);
      if (cur.nblk == 0) {
        if (lane == 0) {
          recs[st].s[0] = SlotRec{0, 0, 0, 0, 0, 0, 0, 1};
          recs[st].s[1] = SlotRec{0, 0, 0, 0, 0, 0, 0, 0};
          mbar_arrive(full);
        }
        ++i;
        return false;
      }
      // the query-operand rows to copy: every active slot's (bf16), or (E4M3)
      // those this stage does not hold yet
      bool needq[2];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        needq[j] = (cur.s[j].flags & F_ACTIVE) != 0;
        if (F8 && needq[j]) needq[j] = qtag[2 * st + j] != cur.s[j].tok * Hkv + cur.s[j].kv;
      }
      const int nq = (needq[0] ? 1 : 0) + (needq[1] ? 1 : 0);
      if (F8 && lane < 16) reinterpret_cast<float*>(gb + M::OFF_INV + st * 64)[lane] = cur.invl;
      __syncwarp();
      if (lane == 0) {
        recs[st].s[0] = cur.s[0];
        recs[st].s[1] = cur.s[1];
        if (F8) {
#pragma unroll
          for (int j = 0; j < 2; ++j)
            if (needq[j]) qtag[2 * st + j] = cur.s[j].tok * Hkv + cur.s[j].kv;
        }
        // per block: K and V (4 KB each bf16, 2 KB each E4M3); per slot
        // copied: its 8 query-operand rows (2 KB)
        mbar_arrive_expect_tx(full, (uint32_t)cur.nblk * (F8 ? 4096u : 8192u) + (uint32_t)nq * 2048u);
      }
      __syncwarp();
      // a decode's newest token, written by the preceding grid, sits in its
      // last block: see that grid's writes before copying such a block
      if (!waited && cur.last_blk) {
        griddep_wait();
        waited = true;
      }
      const uint32_t sbase = base + M::OFF_STAGE + st * M::kStageBytes;
      if (lane < cur.nblk) {
        int pid = cur.pid;
        if (pid < 0 || pid >= p.num_blocks) {
          report_error(p.err, PA_DEVERR_BLOCK_ID, lane);
          pid = 0;
        }
        if constexpr (F8) {
          const int row = (pid * Hkv + cur.kvl) * kBlockSize;  // the block's first row
          tma_load_2d(sbase + lane * 2048, &tp.tm_k, 0, row, full);
          tma_load_2d(sbase + L::kKvTile + lane * 2048, &tp.tm_v, 0, row, full);
        } else {
          const int grp = (pid * Hkv + cur.kvl) * (kBlockSize / 8);  // the block's first 8-key group
          tma_load_4d(sbase + lane * 2 * L::kGroup, &tp.tm_k, 0, 0, 0, grp, full);
          tma_load_4d(sbase + L::kKvTile + lane * 2 * L::kGroup, &tp.tm_v, 0, 0, 0, grp, full);
        }
      }
      if (lane < 2 && (lane == 0 ? needq[0] : needq[1])) {  // the query operand rows of slot `lane`
        const int qtok = lane == 0 ? cur.s[0].tok : cur.s[1].tok;
        const int qkv = lane == 0 ? cur.s[0].kv : cur.s[1].kv;
        // 8 rows from the group's first (rows past the group are other
        // heads' queries, or zeros past the end: they only feed the slot's
        // unused columns)
        tma_load_3d(sbase + 2 * L::kKvTile + lane * 2048, &tp.tm_q, 0, qtok * Hq + qkv * G, 0,
                    full);
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
      mbar_wait_bounded(BAR(M::B_FULL + j % kStages), (uint32_t)(j / kStages) & 1u);
  } else if (warp == 5) {
    // ======================= MMA issuer (lane 0) =======================
    // Two kinds of work, each in tile order: S(j) once tile j has landed and
    // S buffer j % kSP is free (the P.V of tile j - kSP issued, hence its
    // softmax done), and O(j) = P.V once the softmax of tile j is done. Whichever is
    // ready is issued, the P.V first: it frees a stage for the producer. O^T
    // always accumulates: its columns start at zero and an epilogue zeroes a
    // slot's columns after reading them.
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_tc(128, L::kN, false, false, F8);
      constexpr uint32_t id_o = idesc_tc(128, L::kN, true, false, F8);
      // K-major: the K tile and the query operand (8-row groups kGroup apart
      // in the K tile, 2 KB / 1 KB apart in the query operand)
      const uint64_t kdesc = smem_desc_sw128(base, 16, L::kGroup);
      const uint64_t qdesc = smem_desc_sw128(base, 16, F8 ? 1024 : 2048);
      const uint64_t pdesc = smem_desc_sw128(base, 16, 1024);  // K-major: P^T
      // M/N-major: V^T (8-key groups kGroup apart; bf16: the 64-dim halves kHalfOff apart)
      const uint64_t vdesc = smem_desc_sw128(base, F8 ? 16 : L::kHalfOff, L::kGroup);
      constexpr int kSteps = 128 / L::kKStep;  // MMAs per product (K = 128 dims or keys)
      int ns = 0, no = 0;  // next tile for S, next tile for P.V
      bool end_seen = false;
      uint32_t spins = 0;
      uint64_t t0 = 0;
#pragma unroll 1
      while (!(end_seen && no == ns)) {
        if (no < ns && mbar_test(BAR(M::B_PREADY + no % kSP), (uint32_t)(no / kSP) & 1u)) {
          tc_fence_after();
          const int st = no % kStages;
          const uint64_t a0 = vdesc + ((uint64_t)(M::OFF_STAGE + st * M::kStageBytes + L::kKvTile) >> 4);
          const uint64_t b0 = pdesc + ((uint64_t)(M::OFF_P + (no % kSP) * L::kPBytes) >> 4);
#pragma unroll
          for (int ks = 0; ks < kSteps; ++ks) {
            if constexpr (F8) {  // keys 32 ks .. 32 ks + 31: 4 rows of 8-key groups
              umma_e4m3(tmem + M::kTmO, a0 + (uint64_t)((ks * 4 * L::kGroup) >> 4),
                        b0 + (uint64_t)((ks * 32) >> 4), id_o, 1u);
            } else {  // keys 16 ks .. 16 ks + 15: groups 2 ks, 2 ks + 1
              umma_bf16(tmem + M::kTmO, a0 + (uint64_t)((ks * 2 * L::kGroup) >> 4),
                        b0 + (uint64_t)(((ks >> 2) * 2048 + (ks & 3) * 32) >> 4), id_o, 1u);
            }
          }
          umma_commit(BAR(M::B_EMPTY + st));
          umma_commit(BAR(M::B_PFREE + no % kSP));
          ++no;
          spins = 0;
        } else if (!end_seen && ns <= no + kSP - 1 &&
                   mbar_test(BAR(M::B_FULL + ns % kStages), (uint32_t)(ns / kStages) & 1u)) {
          const int st = ns % kStages;
          if (recs[st].s[0].pad) {
            end_seen = true;
          } else {
            tc_fence_after();
            const uint64_t a0 = kdesc + ((uint64_t)(M::OFF_STAGE + st * M::kStageBytes) >> 4);
            const uint64_t b0 =
                qdesc + ((uint64_t)(M::OFF_STAGE + st * M::kStageBytes + 2 * L::kKvTile) >> 4);
#pragma unroll
            for (int ks = 0; ks < kSteps; ++ks) {  // head dims ks * kKStep ..
              if constexpr (F8) {
                umma_e4m3(tmem + M::kTmS + L::kN * (ns % kSP), a0 + (uint64_t)((ks * 32) >> 4),
                          b0 + (uint64_t)((ks * 32) >> 4), id_s, ks > 0 ? 1u : 0u);
              } else {
                umma_bf16(tmem + M::kTmS + L::kN * (ns % kSP),
                          a0 + (uint64_t)(((ks >> 2) * L::kHalfOff + (ks & 3) * 32) >> 4),
                          b0 + (uint64_t)(((ks >> 2) * 1024 + (ks & 3) * 32) >> 4), id_s,
                          ks > 0 ? 1u : 0u);
              }
            }
            umma_commit(BAR(M::B_S + ns % kSP));
            ++ns;
          }
          spins = 0;
        } else if (++spins > 64) {  // nothing ready: give up after PA_WAIT_LIMIT_NS without progress
          if (spins == 65) t0 = global_timer_ns();
          if (global_timer_ns() - t0 > PA_WAIT_LIMIT_NS) {
            report_error(p.err, PA_DEVERR_WAIT_TIMEOUT, 2000 + M::B_PREADY);
            break;
          }
        }
      }
      // every MMA issued above has completed before TMEM is released
      umma_commit(BAR(M::B_DRAIN));
      mbar_wait_bounded(BAR(M::B_DRAIN), 0);
    }
    __syncwarp();
  } else {
    // ======================= softmax + epilogue (warps 0-3) =======================
    const int m = warp * 32 + lane;  // key row of S^T and head dim of O^T: the TMEM lane
    const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
    float* const xch = reinterpret_cast<float*>(gb + M::OFF_XCH);
    int nx = 0;  // exchanges done
    // Per-head max or sum over the 128 softmax threads: warp reduction, then
    // the four warps meet on an mbarrier (bounded wait). Exchange k uses
    // buffer and barrier k % 2: a buffer is rewritten only after every thread
    // has passed the other barrier, i.e. has read this one.
    auto block_reduce = [&](float (&v)[G], bool is_max) -> bool {
      const float x = is_max ? warp_reduce_heads<G, true>(v, lane) : warp_reduce_heads<G, false>(v, lane);
      const int kx = nx++;
      float* const xb = xch + (kx & 1) * 64;
      if (lane < G) xb[warp * 16 + tc_head_of_lane<G>(lane)] = x;
      mbar_arrive(BAR(M::B_XCH + (kx & 1)));
      if (!wait(M::B_XCH + (kx & 1), kx >> 1)) return false;
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float a = xb[h], b = xb[16 + h], c = xb[32 + h], d = xb[48 + h];
        v[h] = is_max ? fmaxf(fmaxf(a, b), fmaxf(c, d)) : (a + b) + (c + d);
      }
      return true;
    };
    // Whether any of the 128 threads holds v, on the same exchange: the
    // warps' votes meet in the exchange buffer.
    auto block_any = [&](bool v, bool& any) -> bool {
      const bool wv = __any_sync(kAllLanes, v);
      const int kx = nx++;
      float* const xb = xch + (kx & 1) * 64;
      if (lane == 0) xb[warp * 16 + 15] = wv ? 1.f : 0.f;
      mbar_arrive(BAR(M::B_XCH + (kx & 1)));
      if (!wait(M::B_XCH + (kx & 1), kx >> 1)) return false;
      any = (xb[15] + xb[31]) + (xb[47] + xb[63]) != 0.f;
      return true;
    };
    // O^T starts at zero (the P.V MMAs always accumulate)
    {
      uint32_t z[8];
#pragma unroll
      for (int c = 0; c < 8; ++c) z[c] = 0u;
#pragma unroll
      for (int c = 0; c < L::kN; c += 8) tm_st<8>(trow + M::kTmO + c, z);
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
    // bf16: P^T[8 slot + h][m] of buffer b: half m / 64, row 8 slot + h,
    // 16-byte unit (m % 64) / 8 swizzled by h
    auto prow = [&](int b, int j, int h) -> uint16_t* {
      return reinterpret_cast<uint16_t*>(gb + M::OFF_P + b * L::kPBytes + (m >> 6) * 2048 +
                                         j * 1024 + h * 128 + ((((m & 63) >> 3) ^ h) << 4) +
                                         (m & 7) * 2);
    };
    // E4M3: P'^T row r = 16 slot + 8 hl + h of buffer b, byte m: 16-byte unit
    // m / 16 swizzled by h
    auto prow8 = [&](int b, int r) -> unsigned char* {
      return gb + M::OFF_P + b * L::kPBytes + r * 128 + ((((m >> 4) ^ (r & 7))) << 4) + (m & 15);
    };
    // This thread's P^T entries of slot j in buffer b: bf16, or (E4M3)
    // P' = 256 p as hi + lo, one byte per row of the slot
    auto write_p = [&](int b, int j, const float (&pr)[G]) {
      if constexpr (F8) {
#pragma unroll
        for (int h = 0; h < G; h += 2) {
          const float x0 = 256.f * pr[h], x1 = h + 1 < G ? 256.f * pr[h + 1] : 0.f;
          const uint16_t hi = float2_to_e4m3x2(x0, x1);
          const float2 hf = e4m3x2_to_float2(hi);
          const uint16_t lo = float2_to_e4m3x2(x0 - hf.x, x1 - hf.y);
          *prow8(b, 16 * j + h) = (unsigned char)(hi & 0xffu);
          *prow8(b, 16 * j + 8 + h) = (unsigned char)(lo & 0xffu);
          if (h + 1 < G) {
            *prow8(b, 16 * j + h + 1) = (unsigned char)(hi >> 8);
            *prow8(b, 16 * j + 8 + h + 1) = (unsigned char)(lo >> 8);
          }
        }
      } else {
#pragma unroll
        for (int h = 0; h < G; ++h) *prow(b, j, h) = bf16_bits(pr[h]);
      }
    };
    // The reference max moves only when a tile's max exceeds it by more than
    // this (log2 units): 2^8 for bf16 P, 0.75 for E4M3 P' = 256 p <= 430.
    constexpr float kSlack = F8 ? 0.75f : 8.f;
    // E4M3: a reference is set 1 (log2 units) above the maxima it is taken
    // from, so it moves only for a score 1.75 above them (P' then peaks at
    // 128 and loses one octave at the bottom, below 2^-16 of the maximum)
    constexpr float kHead = F8 ? 1.f : 0.f;
    auto epilogue = [&](const SlotRec& e0, const SlotRec& e1, int eb, int ei, const float (&em)[2][G],
                        const float (&el)[2][G]) -> bool {
      if (!wait(M::B_PFREE + eb, ei / kSP)) return false;
      tc_fence_after();
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const SlotRec rc = j == 0 ? e0 : e1;
        if (!(rc.flags & F_LAST)) continue;
        float ls[G];
#pragma unroll
        for (int h = 0; h < G; ++h) ls[h] = el[j][h];
        if (!block_reduce(ls, false)) return false;
        const uint32_t ocol = M::kTmO + L::kSlotCols * j;
        float o[G];
        {
          uint32_t oa[G];
          tm_ld<G>(trow + ocol, oa);
          if constexpr (F8) {  // hi + lo groups, back from P' = 256 p
            uint32_t ob[G];
            tm_ld<G>(trow + ocol + 8, ob);
            tmem_wait_ld();
#pragma unroll
            for (int h = 0; h < G; ++h)
              o[h] = (__uint_as_float(oa[h]) + __uint_as_float(ob[h])) * (1.f / 256.f);
          } else {
            tmem_wait_ld();
#pragma unroll
            for (int h = 0; h < G; ++h) o[h] = __uint_as_float(oa[h]);
          }
        }
        if (rc.flags & F_WHOLE) {
          float mh[G];
#pragma unroll
          for (int h = 0; h < G; ++h) mh[h] = em[j][h];
          // Cascade: the prefix partials of this (token, kv head), one per
          // key chunk, folded in by log-sum-exp renormalisation.
#pragma unroll 1
          for (int c = 0; c < p.prefix_chunks; ++c) {
            const float* const sl =
                p.prefix_partials + (((size_t)c * p.num_tokens + rc.tok) * Hkv + rc.kv) * p.slot_floats;
#pragma unroll
            for (int h = 0; h < G; ++h) {
              const float mc = __ldcg(sl + h);
              const float mn = fmaxf(mh[h], mc);
              const float a = exp2f(mh[h] - mn), bb = exp2f(mc - mn);
              ls[h] = ls[h] * a + __ldcg(sl + G + h) * bb;
              o[h] = o[h] * a + __ldcg(sl + 16 + h * kD + m) * bb;
              mh[h] = mn;
            }
          }
          uint16_t* const orow = p.out + ((size_t)rc.tok * Hq + (size_t)rc.kv * G) * kD + m;
#pragma unroll
          for (int h = 0; h < G; ++h) orow[h * kD] = bf16_bits(o[h] * (p.v_scale / ls[h]));
        } else {
          // a partial (m, l, o) for the merge pass in slot u + w: tokens
          // increase with the position order, so the slot is unique per portion
          float* const slot =
              p.partials + (size_t)(rc.tok * Hkv + rc.kv + w) * (size_t)p.slot_floats;
          if (m == 0) {
#pragma unroll
            for (int h = 0; h < G; ++h) {
              __stcg(slot + h, em[j][h]);
              __stcg(slot + G + h, ls[h]);
            }
          }
#pragma unroll
          for (int h = 0; h < G; ++h) __stcg(slot + 16 + h * kD + m, o[h]);
        }
        // the slot's columns start the next portion at zero
        uint32_t z[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) z[c] = 0u;
#pragma unroll
        for (int g = 0; g < L::kSlotCols; g += 8) tm_st<8>(trow + ocol + g, z);
        tmem_wait_st();
      }
      tc_fence_before();  // the next tile's P.V accumulates into O^T
      return true;
    };
    // A tile's epilogue (portions ending there) runs while the next tile is
    // in the softmax, before that tile's P is released to the MMA warp: by
    // then tile i's P.V has usually completed, and the next P.V, which would
    // accumulate into the slot's columns, waits for the epilogue's reads and
    // zeroing. The ending slots' maxima and sums are kept for it. At G = 8
    // (long portions, few epilogues, more registers) it runs right after the
    // tile, once its P.V has completed (measured faster there, slower at G <= 4).
    constexpr bool kDefer = G <= 4;
    bool pend = false;
    SlotRec pr0{0, 0, 0, 0, 0, 0, 0, 0}, pr1{0, 0, 0, 0, 0, 0, 0, 0};
    int pb = 0, pi = 0;
    float pm[2][G], pl[2][G];
    int i = 0;
    bool ok = true;
#pragma unroll 1
    while (ok) {
      const int st = i % kStages;
      if (!wait(M::B_FULL + st, i / kStages)) { ok = false; break; }  // the tile record is visible
      const SlotRec r0 = recs[st].s[0], r1 = recs[st].s[1];
      if (r0.pad) break;
      const int b = i % kSP;  // S^T and P^T buffer of this tile
      if (!wait(M::B_S + b, i / kSP)) { ok = false; break; }
      tc_fence_after();
      // this thread's key: slot my (-1: no key), valid when inside its sequence
      const bool in0 = (r0.flags & F_ACTIVE) && m >= r0.row0 && m < r0.row0 + r0.nrows;
      const bool in1 = (r1.flags & F_ACTIVE) && m >= r1.row0 && m < r1.row0 + r1.nrows;
      const int my = in0 ? 0 : (in1 ? 1 : -1);
      const bool valid = in0 ? (r0.key0 + (m - r0.row0) < r0.len)
                             : (in1 ? (r1.key0 + (m - r1.row0) < r1.len) : false);
      // P^T buffer b is free once the P.V of tile i - kSP has completed
      if (i >= kSP && !wait(M::B_PFREE + b, i / kSP - 1)) { ok = false; break; }
      // One pass per active slot (two only where the tile crosses from one
      // portion into the next): the slot's scores, its maxima, P^T rows.
      const int nact = ((r0.flags & F_ACTIVE) ? 1 : 0) + ((r1.flags & F_ACTIVE) ? 1 : 0);
#pragma unroll 1
      for (int pass = 0; pass < nact; ++pass) {
        const int jj = (pass == 0 && (r0.flags & F_ACTIVE)) ? 0 : 1;
        const int fl = jj ? r1.flags : r0.flags;
        const bool mine = valid && my == jj;  // this thread's key belongs to slot jj
        const uint32_t scol = M::kTmS + L::kN * b + L::kSlotCols * jj;
        float t[G];
        if constexpr (F8) {  // hi and lo column groups, the row scales undone
          uint32_t shi[G], slo[G];
          tm_ld<G>(trow + scol, shi);
          tm_ld<G>(trow + scol + 8, slo);
          tmem_wait_ld();
          const float* const inv = reinterpret_cast<const float*>(gb + M::OFF_INV + st * 64 + jj * 32);
#pragma unroll
          for (int h = 0; h < G; ++h)
            t[h] = mine ? (__uint_as_float(shi[h]) + __uint_as_float(slo[h])) * (inv[h] * p.scale_log2)
                        : -INFINITY;
        } else {
          uint32_t sr[G];
          tm_ld<G>(trow + scol, sr);
          tmem_wait_ld();
#pragma unroll
          for (int h = 0; h < G; ++h) t[h] = mine ? __uint_as_float(sr[h]) * p.scale_log2 : -INFINITY;
        }
        float mr[G], lt[G];
#pragma unroll
        for (int h = 0; h < G; ++h) {
          mr[h] = jj ? mref[1][h] : mref[0][h];
          lt[h] = jj ? lth[1][h] : lth[0][h];
        }
        // Reference maxima: a portion's first tile sets them (it holds the
        // portion's first key, so they are finite); later tiles move them
        // only by more than kSlack, rescaling the slot's O^T columns. Where
        // that is rare (bf16: P up to 2^8; E4M3 at G = 8) the threads first
        // vote on whether any score is above its reference by that much, and
        // only a tile the vote flags takes its maxima. (E4M3's slack is small:
        // on the Llama-8B batch at G = 4 about one tile in four moves its
        // reference, and the vote then costs a second exchange.)
        constexpr bool kVote = !F8 || G == 8;
        const bool first = (fl & F_FIRST) != 0;
        bool need_max = first || !kVote;
        if (!need_max) {
          bool over = false;
#pragma unroll
          for (int h = 0; h < G; ++h) over |= t[h] > mr[h] + kSlack;
          if (!block_any(over, need_max)) { ok = false; break; }
        }
        if (need_max) {
          float tm[G];
#pragma unroll
          for (int h = 0; h < G; ++h) tm[h] = t[h];
          if (!block_reduce(tm, true)) { ok = false; break; }
          bool resc = false;
          float alpha[G];
#pragma unroll
          for (int h = 0; h < G; ++h) {
            alpha[h] = 1.f;
            if (first) {
              mr[h] = tm[h] + kHead;
              lt[h] = 0.f;
            } else if (tm[h] > mr[h] + kSlack) {
              alpha[h] = exp2f(mr[h] - (tm[h] + kHead));
              mr[h] = tm[h] + kHead;
              resc = true;
            }
          }
          if (resc) {  // uniform: every thread holds the same maxima
            // O^T is stable once the previous tile's P.V has completed
            if (!wait(M::B_PFREE + (i - 1) % kSP, (i - 1) / kSP)) { ok = false; break; }
            tc_fence_after();
            const uint32_t ocol = M::kTmO + L::kSlotCols * jj;
#pragma unroll
            for (int g = 0; g < L::kSlotCols; g += 8) {  // E4M3: the hi and the lo group
              uint32_t o[G];
              tm_ld<G>(trow + ocol + g, o);
              tmem_wait_ld();
#pragma unroll
              for (int h = 0; h < G; ++h) o[h] = __float_as_uint(__uint_as_float(o[h]) * alpha[h]);
              tm_st<G>(trow + ocol + g, o);
            }
            tmem_wait_st();
#pragma unroll
            for (int h = 0; h < G; ++h) lt[h] *= alpha[h];
          }
        }
        float pr[G];
#pragma unroll
        for (int h = 0; h < G; ++h) pr[h] = mine ? ex2_approx(t[h] - mr[h]) : 0.f;
        write_p(b, jj, pr);
#pragma unroll
        for (int h = 0; h < G; ++h) {
          lt[h] += pr[h];
          if (jj) {
            mref[1][h] = mr[h];
            lth[1][h] = lt[h];
          } else {
            mref[0][h] = mr[h];
            lth[0][h] = lt[h];
          }
        }
        dirty |= 1 << (2 * b + jj);
        if (nact == 1 && (dirty & (1 << (2 * b + (1 - jj))))) {  // the idle slot's rows to zero
          if constexpr (F8) {
#pragma unroll
            for (int h = 0; h < G; ++h) {
              *prow8(b, 16 * (1 - jj) + h) = 0;
              *prow8(b, 16 * (1 - jj) + 8 + h) = 0;
            }
          } else {
#pragma unroll
            for (int h = 0; h < G; ++h) *prow(b, 1 - jj, h) = 0;
          }
          dirty &= ~(1 << (2 * b + (1 - jj)));
        }
      }
      if (!ok) break;
      if (!valid) {
        // A key past the sequence end (or a block slot this tile did not
        // load) has P = 0, but its V row may hold anything, NaN included, and
        // 0 * NaN would poison O: clear the row.
        if constexpr (F8) {
          unsigned char* const vrow = gb + M::OFF_STAGE + st * M::kStageBytes + L::kKvTile + m * 128;
#pragma unroll
          for (int q = 0; q < 8; ++q) *reinterpret_cast<uint4*>(vrow + q * 16) = make_uint4(0u, 0u, 0u, 0u);
        } else {
          unsigned char* const vrow = gb + M::OFF_STAGE + st * M::kStageBytes + L::kKvTile +
                                      (m >> 3) * L::kGroup + (m & 7) * 128;
#pragma unroll
          for (int c = 0; c < 2; ++c)
#pragma unroll
            for (int q = 0; q < 8; ++q)
              *reinterpret_cast<uint4*>(vrow + c * L::kHalfOff + q * 16) = make_uint4(0u, 0u, 0u, 0u);
        }
      }
      fence_proxy_async_smem();  // generic-proxy stores -> visible to the tensor core
      if (pend) {  // the previous tile's epilogue, before this tile's P.V may start
        if (!epilogue(pr0, pr1, pb, pi, pm, pl)) { ok = false; break; }
        pend = false;
      }
      tc_fence_before();
      mbar_arrive(BAR(M::B_PREADY + b));
      if (((r0.flags | r1.flags) & F_LAST) && !kDefer) {  // the epilogue now
        if (!epilogue(r0, r1, b, i, mref, lth)) { ok = false; break; }
      } else if ((r0.flags | r1.flags) & F_LAST) {
        pend = true;
        pr0 = r0;
        pr1 = r1;
        pb = b;
        pi = i;
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
          for (int h = 0; h < G; ++h) {
            pm[j][h] = mref[j][h];
            pl[j][h] = lth[j][h];
          }
      }
      ++i;
    }
    if (ok && pend) epilogue(pr0, pr1, pb, pi, pm, pl);  // the last tile's
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
  // overlapped mixed batch: complete only after the prefill-chunk grid, so
  // that whoever waits for this grid (the merge pass, later work on the
  // stream) sees the whole call
  if (p.overlap && threadIdx.x == 0) griddep_wait();
}

// One warp per (token, kv head): each of the G query rows is scaled by the
// power of two 2^e that brings its largest magnitude into [128, 256) and
// split into E4M3 terms hi = E4M3(x 2^e), lo = E4M3(x 2^e - hi). A bf16 x has
// 8 significant bits, hi takes the top 4 and the remainder fits lo exactly
// unless it falls below E4M3's subnormal step (elements 2^-9 times the row's
// largest or smaller). Rows hi ‖ lo (2 x 128 B) go to qsplit, 2^-e to qinv
// (8 floats per group; unused ones 0).
template <int G>
__global__ void __launch_bounds__(256) pa_qsplit_kernel(const DecodeParams p) {
  griddep_launch_dependents();  // the split-KV grid may start its prologue
  const int grp = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (grp < p.num_tokens * p.num_kv_heads) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const size_t row = (size_t)grp * G + h;  // token * Hq + kv * G + h
      const uint2 raw4 = __ldg(reinterpret_cast<const uint2*>(p.q + row * kD) + lane);
      const float2 a = bf16x2_to_float2(raw4.x), c = bf16x2_to_float2(raw4.y);
      float mx = fmaxf(fmaxf(fabsf(a.x), fabsf(a.y)), fmaxf(fabsf(c.x), fabsf(c.y)));
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(kAllLanes, mx, o));
      // e = 7 - floor(log2 mx), from the exponent field (a zero row keeps e = 0)
      int ex = 0;
      if (mx > 0.f) {
        ex = 7 - (((int)(__float_as_uint(mx) >> 23) & 0xff) - 127);
        ex = ex < -120 ? -120 : (ex > 120 ? 120 : ex);
      }
      const float sc = __uint_as_float((uint32_t)(127 + ex) << 23);   // 2^e, exact
      const float isc = __uint_as_float((uint32_t)(127 - ex) << 23);  // 2^-e
      const float x0 = a.x * sc, x1 = a.y * sc, x2 = c.x * sc, x3 = c.y * sc;
      const uint16_t h01 = float2_to_e4m3x2(x0, x1), h23 = float2_to_e4m3x2(x2, x3);
      const float2 f01 = e4m3x2_to_float2(h01), f23 = e4m3x2_to_float2(h23);
      const uint16_t l01 = float2_to_e4m3x2(x0 - f01.x, x1 - f01.y);
      const uint16_t l23 = float2_to_e4m3x2(x2 - f23.x, x3 - f23.y);
      unsigned char* const dst = const_cast<unsigned char*>(p.qsplit) + row * 2 * kD;
      reinterpret_cast<uint32_t*>(dst)[lane] = (uint32_t)h01 | ((uint32_t)h23 << 16);
      reinterpret_cast<uint32_t*>(dst + kD)[lane] = (uint32_t)l01 | ((uint32_t)l23 << 16);
      if (lane == 0) const_cast<float*>(p.qinv)[(size_t)grp * 8 + h] = isc;
    }
    if (lane >= G && lane < 8) const_cast<float*>(p.qinv)[(size_t)grp * 8 + lane] = 0.f;
  }
  // complete only after the preceding grid (the KV write, the planner or the
  // prefill grid): a dependent that waits for this grid sees theirs too
  griddep_wait();
}

// ---------------------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------------------
namespace {

template <int G, bool F8>
cudaError_t launch_tc_t(const DecodeParams& d, int grid, cudaStream_t s) {
  TcDecodeParams tp;
  tp.d = d;
  const uint64_t qrows = (uint64_t)d.num_tokens * (uint64_t)d.num_q_heads;
  if constexpr (F8) {
    // q' rows as {128 B, rows (256 B apart), hi / lo (128 B apart)}: a box of 8
    // rows lands as [hi, lo][8 rows][128 B]
    const uint64_t qd[3] = {128, qrows, 2}, qs[2] = {2 * kD, kD};
    const uint32_t qb[3] = {128, 8, 2};
    const uint64_t rows = (uint64_t)d.num_blocks * (uint64_t)d.num_kv_heads * kBlockSize;
    const uint64_t cd[2] = {128, rows}, cs[1] = {kD};
    const uint32_t cb[2] = {128, kBlockSize};
    if (!encode_tmap_u8(&tp.tm_q, 3, d.qsplit, qd, qs, qb) ||
        !encode_tmap_u8(&tp.tm_k, 2, d.k_cache, cd, cs, cb) ||
        !encode_tmap_u8(&tp.tm_v, 2, d.v_cache, cd, cs, cb))
      return cudaErrorInvalidValue;
  } else {
    // q as {64 dims, rows, 2 halves}: a box of 8 rows lands as [half][8 rows][128 B]
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
  }
  auto kern = pa_decode_tc_kernel<G, F8>;
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, TcSmem<F8>::SMEM);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = TcSmem<F8>::SMEM;
  cfg.stream = s;
  // Programmatic launch: the grid starts when the preceding grid triggers
  // (the KV write or the query split at its top for a self-planned batch;
  // otherwise the planner or the tensor-core prefill grid, at their end).
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tp);
}

template <int G>
cudaError_t launch_qsplit_t(const DecodeParams& d, cudaStream_t s) {
  const int groups = d.num_tokens * d.num_kv_heads;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((groups + 7) / 8));
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, pa_qsplit_kernel<G>, d);
}

}  // namespace

int decode_tc_workers(int num_sms) {
  return num_sms < kMaxDecodeWorkers ? num_sms : kMaxDecodeWorkers;
}

bool decode_tc_supported(int head_dim, int group, bool f8, int key_start_blocks) {
  (void)key_start_blocks;  // a cascade's suffix pass (bf16 only: no E4M3 cascade)
  return head_dim == kD && !(f8 && key_start_blocks > 0) &&
         (group == 1 || group == 2 || group == 4 || group == 8);
}

cudaError_t launch_decode_tc(const DecodeParams& p, int group, bool f8, int num_sms,
                             cudaStream_t s, int* workers_out) {
  const int grid = decode_tc_workers(num_sms);
  *workers_out = grid;
  switch (group) {
    case 1: return f8 ? launch_tc_t<1, true>(p, grid, s) : launch_tc_t<1, false>(p, grid, s);
    case 2: return f8 ? launch_tc_t<2, true>(p, grid, s) : launch_tc_t<2, false>(p, grid, s);
    case 4: return f8 ? launch_tc_t<4, true>(p, grid, s) : launch_tc_t<4, false>(p, grid, s);
    case 8: return f8 ? launch_tc_t<8, true>(p, grid, s) : launch_tc_t<8, false>(p, grid, s);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_qsplit(const DecodeParams& p, int group, cudaStream_t s) {
  switch (group) {
    case 1: return launch_qsplit_t<1>(p, s);
    case 2: return launch_qsplit_t<2>(p, s);
    case 4: return launch_qsplit_t<4>(p, s);
    case 8: return launch_qsplit_t<8>(p, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace pa
