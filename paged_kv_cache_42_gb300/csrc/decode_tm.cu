// Split-KV paged decode over an E4M3 cache on the tensor cores, one 16-key
// block of ALL eight KV heads per tile ("token-major" tiles).
//
// What is computed is what the other split-KV kernels compute ("vLLM v1 Deep
// Dive: How LLM(...) and the Server Boot and Generate", Part 3, "Aside - KV
// cache and prefix caching": a decode query attends to all of its request's
// blocks; "vLLM: An Exhaustive Technical Study for Kernel Engineers", 2.4:
// the query heads of a KV head share its K/V; 2.8: E4M3 codes with
// per-tensor k_scale / v_scale). The difference is the tile. The cache keeps
// a block's eight KV heads contiguous ([block][kv head][16 keys][128 B]), so
// one 16 KB tensor copy lands K (and one more V) for all of them: 128 rows,
// row = 16 kv + key. Per tile the producer issues two copies instead of
// sixteen, and each KV head's 16 keys sit in one half-warp of the softmax, so
// a head's maxima and sums are taken by shuffles, without a cross-warp
// exchange.
//
// Work. The flattened positions are (token, 16-key block): a token's blocks
// in order, tokens in order; workers (one CTA each: two per SM at G <= 4,
// one at G = 8) take equal contiguous slices. A tile is one position. A
// token split between workers leaves an fp32 partial per KV head, in slot
// (token + worker) * 8 + kv head: token + worker grows by one at every token
// or worker change along the positions, so the slot is unique; the merge
// pass folds them.
//
// Products (tcgen05.mma kind::f8f6f4 on the cached codes):
//   S^T = K Q'^T   M = 128 rows (8 KV heads x 16 keys), N = 2 Hq: the token's
//                  query rows, each scaled by 2^e and split into E4M3 hi and
//                  lo terms by the query-split pass (hi rows, then lo rows);
//                  K = 128 dims. Only the Hq / 8 columns of a row's own KV
//                  head are used.
//   O^T += V^T P'^T  M = 128 dims, N = 2 Hq, K = 128 rows. P'^T is
//                  block-diagonal: row c (query head h, hi or lo) holds
//                  P' = 256 p of the keys of h's KV head and zeros elsewhere,
//                  so each query head sums its own KV head's V rows only. The
//                  zeros are written once; a tile writes its diagonal.
// O^T lives in TMEM in two buffers that alternate per token: a token's first
// P.V overwrites its buffer (no zeroing), and a token's epilogue reads its
// buffer while the next token accumulates in the other.
//
// Softmax (warps 0-3; thread m = TMEM lane m: KV head m / 16, key m % 16).
// Each thread takes its key's score for the G query heads of its KV head,
// (S_hi + S_lo) 2^-e scale log2(e). A token's first tile sets each query
// head's reference 3 above its 16 keys' max; later, a reference moves only
// when a score exceeds it by more than 0.75, and is then set 1 above the
// half-warp's max (so P' <= 430 < 448): a reference only moves in its own
// half-warp. Moving it rescales that head's columns of O^T, which every
// thread holds a row of, so each tile the warps post which heads moved
// (alphas, a flag per warp) on an mbarrier exchange as soon as they know,
// compute P' meanwhile, and collect before releasing P'; a flagged tile
// rescales O^T through TMEM first. Sums stay per thread until the token's
// epilogue (one exchange per token for the heads' sums and maxima).
//
// Roles (192 threads per CTA): warps 0-3 softmax and epilogue, warp 4
// the producer (walks the work list, one record per tile, two or three tensor
// copies), warp 5 allocates TMEM and one thread issues the MMAs. Every wait
// is bounded; one that gives up sets the device error word.
#include <cuda.h>
#include <cuda_bf16.h>

#include "pa_internal.h"
#include "ptx.cuh"

namespace pa {

namespace {

// References (log2 units) are set this far above the maxima they come from:
// a token's first, from one block's 16 keys, PA_TM_HEAD_FIRST (about the
// growth of the maximum from 16 keys to a few thousand, so the reference
// seldom moves again); a moved one PA_TM_HEAD. P' then peaks at 256 x 2^-head
// and keys 2^-(17 - head) below the reference fall under E4M3's subnormal
// step. Measured on the Llama-8B batch: first / moved headroom 1 / 1
// 64.3 us, 2 / 2 60.9 us, 3 / 1 59.0 us, 3 / 3 59.0 us, 2.5 / 1 60.2 us.
#ifndef PA_TM_HEAD
#define PA_TM_HEAD 1.f
#endif
#ifndef PA_TM_HEAD_FIRST
#define PA_TM_HEAD_FIRST 3.f
#endif

constexpr unsigned kLanes = 0xffffffffu;
constexpr int kTmD = 128;    // head dim
constexpr int kTmHkv = 8;    // KV heads: 8 x 16 keys = the MMA's 128 rows
constexpr int kTmThreads = 192;

template <int G, int CPS>
struct TmL {
  static constexpr int HQ = kTmHkv * G;          // query heads of a token
  static constexpr int N = 2 * HQ;               // MMA N: hi rows, then lo rows
  // CTAs resident per SM: two (G <= 4) take two stages each, so an SM holds
  // the same bytes in flight in two independent per-tile chains
  static constexpr int kStages = CPS == 2 ? 2 : (G == 8 ? 3 : 4);
  static constexpr int kKvTile = 16384;          // one block, all KV heads: [128 rows][128 B]
  static constexpr int kQBytes = N * 128;        // a token's q' rows: [hi, lo][HQ rows][128 B]
  static constexpr int kStageBytes = 2 * kKvTile + kQBytes;
  static constexpr int kPBytes = N * 128;        // P'^T: [N rows][128 keys]
  static constexpr int OFF_STAGE = 0;
  static constexpr int OFF_P = kStages * kStageBytes;  // two P'^T buffers
  static constexpr int OFF_REC = OFF_P + 2 * kPBytes;  // a 32-byte record per stage
  static constexpr int OFF_INV = OFF_REC + kStages * 32;   // per stage: 2^-e of the HQ rows
  static constexpr int OFF_QTAG = OFF_INV + kStages * HQ * 4;  // token whose q' a stage holds
  // exchange, two buffers: [4 warp flags][HQ alphas][HQ sums][HQ maxima] floats
  static constexpr int XCH_FLOATS = 4 + 3 * HQ;
  static constexpr int OFF_XCH = (OFF_QTAG + kStages * 4 + 15) / 16 * 16;
  static constexpr int OFF_BAR = (OFF_XCH + 2 * XCH_FLOATS * 4 + 7) / 8 * 8;
  // barriers: FULL[stages], EMPTY[stages], S[2], P_READY[2], P_FREE[2], XCH[2], DRAIN
  static constexpr int B_FULL = 0, B_EMPTY = kStages, B_S = 2 * kStages, B_PREADY = B_S + 2,
                       B_PFREE = B_S + 4, B_XCH = B_S + 6, B_DRAIN = B_S + 8,
                       B_COUNT = B_DRAIN + 1;
  static constexpr int OFF_TSLOT = OFF_BAR + 8 * B_COUNT;
  static constexpr int OFF_UNITS = (OFF_TSLOT + 16 + 15) / 16 * 16;  // self-planned unit table
  static constexpr int SMEM = OFF_UNITS + (int)sizeof(UnitInfo) * (kSelfPlanMaxReqs + 1) + 1024;
  static_assert(CPS == 1 || CPS == 2, "one or two CTAs per SM");
  // 228 KB of shared memory per SM, 1 KB of it reserved per resident CTA
  static_assert(SMEM <= (CPS == 1 ? 227 * 1024 : 113 * 1024), "CTAs per SM fit in shared memory");
  static_assert(kStageBytes % 1024 == 0 && kPBytes % 1024 == 0, "1024-byte aligned operand tiles");
  // TMEM columns: S^T buffers at 0 and N, O^T buffers at 2N and 3N
  static constexpr uint32_t kTmemCols = 4 * N;
  static_assert(CPS * kTmemCols <= 512, "the resident CTAs' TMEM fits in 512 columns");
  static constexpr int CW = HQ < 16 ? HQ : 16;  // O^T columns per TMEM load in epilogues
};

// Tile record flags.
constexpr int T_FIRST = 1;  // the token's first tile in this CTA
constexpr int T_LAST = 2;   // the token's last tile in this CTA
constexpr int T_WHOLE = 4;  // the CTA holds all of the token's blocks: store bf16 output
constexpr int T_PAR = 8;    // O^T buffer 1 (else 0)
constexpr int T_END = 16;   // no more tiles
struct TmRec {
  int tok, len, key0, flags;  // key0: the block's first key
  int pad[4];
};
static_assert(sizeof(TmRec) == 32, "records are 32 bytes");

// Max or sum over the 16 lanes of a half-warp (every lane gets the result).
__device__ __forceinline__ float half_max(float v) {
#pragma unroll
  for (int o = 1; o < 16; o <<= 1) v = fmaxf(v, __shfl_xor_sync(kLanes, v, o));
  return v;
}
__device__ __forceinline__ float half_sum(float v) {
#pragma unroll
  for (int o = 1; o < 16; o <<= 1) v += __shfl_xor_sync(kLanes, v, o);
  return v;
}

}  // namespace

struct TmDecodeParams {
  // q' rows as {128 B, T * Hq rows, 2 (hi, lo)}, box {128, Hq, 2}; a cache as
  // {128 B, blocks * 8 * 16 rows}, box {128, 128}
  CUtensorMap tm_q;
  CUtensorMap tm_k;
  CUtensorMap tm_v;
  DecodeParams d;
};

template <int G, int CPS>
__global__ void __launch_bounds__(kTmThreads, CPS)
    pa_decode_tm_kernel(const __grid_constant__ TmDecodeParams tp) {
  using L = TmL<G, CPS>;
  constexpr int HQ = L::HQ, N = L::N, kStages = L::kStages;
  const DecodeParams& p = tp.d;
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  unsigned char* const gb = smem_raw + (base - raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the merge pass may be placed as CTAs of this grid retire
  griddep_launch_dependents();
  auto BAR = [&](int i) -> uint32_t { return base + L::OFF_BAR + 8u * (uint32_t)i; };
  auto wait = [&](int i, int parity) -> bool {
    if (mbar_wait_bounded(BAR(i), (uint32_t)parity & 1u)) return true;
    report_error(p.err, PA_DEVERR_WAIT_TIMEOUT, 3000 + i);
    return false;
  };
  TmRec* const recs = reinterpret_cast<TmRec*>(gb + L::OFF_REC);

  if (threadIdx.x == 0) {
    for (int i = 0; i < L::B_COUNT; ++i) {
      // P_READY and the exchanges: the 128 softmax threads; the rest once
      const bool by_softmax = i == L::B_PREADY || i == L::B_PREADY + 1 || i == L::B_XCH ||
                              i == L::B_XCH + 1;
      mbar_init(BAR(i), by_softmax ? 128 : 1);
    }
    fence_barrier_init();
  }
  // P'^T starts at zero: off its diagonal it stays zero
  for (int idx = threadIdx.x; idx < (2 * L::kPBytes) / 16; idx += kTmThreads)
    reinterpret_cast<uint4*>(gb + L::OFF_P)[idx] = make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async_smem();
  if (warp == 5) {
    tmem_alloc(base + L::OFF_TSLOT, L::kTmemCols);
    tmem_relinquish();
  }

  // The work list: the planner's (one unit per token, positions = its
  // blocks), or built here for a decode-only batch.
  const UnitInfo* units = p.units;
  int W, K;
  if (p.self_plan) {
    UnitInfo* const su = reinterpret_cast<UnitInfo*>(gb + L::OFF_UNITS);
    __shared__ int s_tot[kTmThreads / 32];
    const int R = p.num_reqs, T = p.num_tokens;
    int carry = 0;
    for (int r0 = 0; r0 < R; r0 += kTmThreads) {
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
          n = (Lr + kBlockSize - 1) / kBlockSize;
        }
      }
      int incl = n;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(kLanes, incl, o);
        if (lane >= o) incl += y;
      }
      if (lane == 31) s_tot[warp] = incl;
      __syncthreads();
      int off = carry;
      for (int w2 = 0; w2 < warp; ++w2) off += s_tot[w2];
      if (r < R) su[r] = UnitInfo{q0, r, n > 0 ? Lr : 0, off + incl - n};
      for (int w2 = 0; w2 < kTmThreads / 32; ++w2) carry += s_tot[w2];
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
    griddep_wait();  // the plan (the query split before this grid waited for it)
    W = __ldcg(&p.header->num_positions);
    K = __ldcg(&p.header->num_units);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(gb + L::OFF_TSLOT);

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
      const int4 u = p.self_plan ? *reinterpret_cast<const int4*>(units + k)
                                 : __ldcg(reinterpret_cast<const int4*>(units + k));
      return UnitInfo{u.x, u.y, u.z, u.w};
    };
    // the walk: position y is block blk of the nb blocks of unit k (a token);
    // np counts the tokens this CTA has started, pstart is the first block of
    // the current one in this slice
    int k = 0;
    UnitInfo U{0, 0, 0, 0}, Un{0, 0, 0, 0};
    int nb = 1, blk = 0, y = S, pstart = 0, np = 0;
    bool pfirst = true;
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
        const unsigned bal = __ballot_sync(kLanes, ok);
        lo = lo + (31 - __clz(bal)) * step;
        hi = min(hi, lo + step);
      }
      k = lo;
      U = load_unit(k);
      Un = load_unit(k + 1);
      nb = max(1, (U.len + kBlockSize - 1) / kBlockSize);
      blk = S - U.base;
      pstart = blk;
      if (w > 0 && lane == 0) {  // the merge task of the slice boundary before this worker
        int4 task = make_int4(-1, 0, 0, 0);
        if (blk != 0) {
          const int first = S - blk;
          const int wf = worker_of(first, W, NW);
          if (w == wf + 1) task = make_int4(U.tok, 0, wf, worker_of(first + nb - 1, W, NW));
        }
        p.merge_tasks[w] = task;
      }
    }
    // The split query rows and scales, and the K/V write before them, come
    // from the preceding grids: a planned batch waited for them at the top; a
    // self-planned one waits below, after the K/V copies of its first two
    // tiles that the write does not touch.
    bool waited = !p.self_plan;

    struct Meta {
      TmRec r;
      int live;      // 0: no more tiles
      int lastblk;   // the token's last block (it holds the newest key)
      int pid;       // lane 0: the block id (loaded two tiles ahead of its copy)
      float inv0, inv1;  // lanes: 2^-e of query rows lane and lane + 32
    };
    auto load_inv = [&](Meta& t) {  // query row kv * G + g's scale: qinv[(token * 8 + kv) * 8 + g]
      const size_t qb = (size_t)t.r.tok * kTmHkv * 8;
      if (lane < HQ) t.inv0 = __ldg(p.qinv + qb + (lane / G) * 8 + (lane % G));
      if (lane + 32 < HQ) t.inv1 = __ldg(p.qinv + qb + ((lane + 32) / G) * 8 + ((lane + 32) % G));
    };
    auto next_tile = [&]() -> Meta {
      Meta t;
      t.r = TmRec{0, 0, 0, T_END, {0, 0, 0, 0}};
      t.live = 0;
      t.lastblk = 0;
      t.pid = 0;
      t.inv0 = t.inv1 = 0.f;
      if (y >= E) return t;
      const bool last = blk + 1 == nb || y + 1 == E;
      t.r = TmRec{U.tok, U.len, blk * kBlockSize,
                  (pfirst ? T_FIRST : 0) | (last ? T_LAST : 0) |
                      ((last && blk + 1 == nb && pstart == 0) ? T_WHOLE : 0) |
                      ((np & 1) ? T_PAR : 0),
                  {0, 0, 0, 0}};
      t.live = 1;
      t.lastblk = blk + 1 == nb;
      if (lane == 0) t.pid = __ldg(p.block_tables + (size_t)U.req * p.bt_stride + blk);
      if (waited) load_inv(t);
      pfirst = false;
      ++y;
      ++blk;
      if (blk == nb && y < E) {  // on to the next token with keys
        do {
          ++k;
          U = Un;
          Un = load_unit(k + 1);
        } while (U.len <= 0);
        nb = max(1, (U.len + kBlockSize - 1) / kBlockSize);
        blk = 0;
        pstart = 0;
        pfirst = true;
        ++np;
      }
      return t;
    };

    int i = 0;
    int* const qtag = reinterpret_cast<int*>(gb + L::OFF_QTAG);
    if (lane < kStages) qtag[lane] = -1;
    __syncwarp();
    auto block_id = [&](const Meta& t) -> int {
      int pid = t.pid;
      if (pid < 0 || pid >= p.num_blocks) {
        report_error(p.err, PA_DEVERR_BLOCK_ID, t.r.key0 / kBlockSize);
        pid = 0;
      }
      return pid;
    };
    bool pre0 = false, pre1 = false;  // tiles 0 and 1: K/V copies already issued
    auto issue = [&](const Meta& cur, Meta& nxt2) -> bool {  // false: stop
      nxt2 = next_tile();
      const int st = i % kStages;
      if (i >= kStages && !wait(L::B_EMPTY + st, (i / kStages) - 1)) return false;
      const uint32_t full = BAR(L::B_FULL + st);
      if (!cur.live) {
        if (lane == 0) {
          recs[st] = cur.r;  // T_END
          mbar_arrive(full);
        }
        ++i;
        return false;
      }
      const bool needq = qtag[st] != cur.r.tok;
      float* const inv = reinterpret_cast<float*>(gb + L::OFF_INV + st * HQ * 4);
      if (lane < HQ) inv[lane] = cur.inv0;
      if (lane + 32 < HQ) inv[lane + 32] = cur.inv1;
      __syncwarp();
      if (lane == 0) {
        recs[st] = cur.r;
        if (needq) qtag[st] = cur.r.tok;
        const bool kv_done = (i == 0 && pre0) || (i == 1 && pre1);
        mbar_arrive_expect_tx(full, (kv_done ? 0u : 2u * L::kKvTile) +
                                        (needq ? (uint32_t)L::kQBytes : 0u));
        const uint32_t sbase = base + L::OFF_STAGE + st * L::kStageBytes;
        if (!kv_done) {
          const int pid = block_id(cur);
          tma_load_2d(sbase, &tp.tm_k, 0, pid * kTmHkv * kBlockSize, full);
          tma_load_2d(sbase + L::kKvTile, &tp.tm_v, 0, pid * kTmHkv * kBlockSize, full);
        }
        if (needq) tma_load_3d(sbase + 2 * L::kKvTile, &tp.tm_q, 0, cur.r.tok * HQ, 0, full);
      }
      __syncwarp();
      ++i;
      return true;
    };
    Meta ma = next_tile();
    Meta mb = next_tile();
    if (!waited) {
      // the first two tiles' K and V (stages 0 and 1), unless they hold a
      // token's newest key
      auto pre_issue = [&](const Meta& t, int j) -> bool {
        if (!t.live || t.lastblk) return false;
        if (lane == 0) {
          const uint32_t full = BAR(L::B_FULL + j);
          const uint32_t sbase = base + L::OFF_STAGE + j * L::kStageBytes;
          const int pid = block_id(t);
          mbar_expect_tx(full, 2u * L::kKvTile);
          tma_load_2d(sbase, &tp.tm_k, 0, pid * kTmHkv * kBlockSize, full);
          tma_load_2d(sbase + L::kKvTile, &tp.tm_v, 0, pid * kTmHkv * kBlockSize, full);
        }
        return true;
      };
      pre0 = pre_issue(ma, 0);
      pre1 = pre_issue(mb, 1);
      griddep_wait();
      waited = true;
      if (ma.live) load_inv(ma);
      if (mb.live) load_inv(mb);
    }
    Meta mc;
#pragma unroll 1
    while (issue(ma, mc) && issue(mb, ma) && issue(mc, mb)) {
    }
    // every copy issued has landed before the CTA may exit
    for (int j = i > kStages ? i - kStages : 0; j < i; ++j)
      mbar_wait_bounded(BAR(L::B_FULL + j % kStages), (uint32_t)(j / kStages) & 1u);
  } else if (warp == 5) {
    // ======================= MMA issuer (lane 0) =======================
    // S(j) once tile j has landed and S buffer j % 2 is free (the P.V of tile
    // j - 2 issued, hence its softmax done); O(j) = P.V once tile j's softmax
    // is done, into the token's O^T buffer, overwriting it at the token's
    // first tile. Whichever is ready is issued, the P.V first.
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_tc(128, N, false, false, true);
      constexpr uint32_t id_o = idesc_tc(128, N, true, false, true);
      const uint64_t kdesc = smem_desc_sw128(base, 16, 1024);  // K-major: K tile, q' rows, P'^T
      const uint64_t vdesc = smem_desc_sw128(base, 16, 1024);  // M/N-major: V^T
      int ns = 0, no = 0;
      bool end_seen = false;
      uint32_t spins = 0;
      uint64_t t0 = 0;
#pragma unroll 1
      while (!(end_seen && no == ns)) {
        if (no < ns && mbar_test(BAR(L::B_PREADY + (no & 1)), (uint32_t)(no >> 1) & 1u)) {
          tc_fence_after();
          const int st = no % kStages;
          const int fl = recs[st].flags;
          const uint32_t od = tmem + 2u * N + ((fl & T_PAR) ? (uint32_t)N : 0u);
          const uint64_t a0 =
              vdesc + ((uint64_t)(L::OFF_STAGE + st * L::kStageBytes + L::kKvTile) >> 4);
          const uint64_t b0 = kdesc + ((uint64_t)(L::OFF_P + (no & 1) * L::kPBytes) >> 4);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)  // rows 32 ks .. 32 ks + 31: four 8-row groups of V
            umma_e4m3(od, a0 + (uint64_t)((ks * 4 * 1024) >> 4), b0 + (uint64_t)((ks * 32) >> 4),
                      id_o, (ks > 0 || !(fl & T_FIRST)) ? 1u : 0u);
          umma_commit(BAR(L::B_EMPTY + st));
          umma_commit(BAR(L::B_PFREE + (no & 1)));
          ++no;
          spins = 0;
        } else if (!end_seen && ns <= no + 1 &&
                   mbar_test(BAR(L::B_FULL + ns % kStages), (uint32_t)(ns / kStages) & 1u)) {
          const int st = ns % kStages;
          if (recs[st].flags & T_END) {
            end_seen = true;
          } else {
            tc_fence_after();
            const uint32_t sbase = L::OFF_STAGE + st * L::kStageBytes;
            const uint64_t a0 = kdesc + ((uint64_t)sbase >> 4);
            const uint64_t b0 = kdesc + ((uint64_t)(sbase + 2 * L::kKvTile) >> 4);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)  // head dims 32 ks .. 32 ks + 31
              umma_e4m3(tmem + (uint32_t)(N * (ns & 1)), a0 + (uint64_t)((ks * 32) >> 4),
                        b0 + (uint64_t)((ks * 32) >> 4), id_s, ks > 0 ? 1u : 0u);
            umma_commit(BAR(L::B_S + (ns & 1)));
            ++ns;
          }
          spins = 0;
        } else if (++spins > 64) {  // nothing ready: give up after PA_WAIT_LIMIT_NS without progress
          if (spins == 65) t0 = global_timer_ns();
          if (global_timer_ns() - t0 > PA_WAIT_LIMIT_NS) {
            report_error(p.err, PA_DEVERR_WAIT_TIMEOUT, 3000 + L::B_PREADY);
            break;
          }
        }
      }
      // every MMA issued above has completed before TMEM is released
      umma_commit(BAR(L::B_DRAIN));
      mbar_wait_bounded(BAR(L::B_DRAIN), 0);
    }
    __syncwarp();
  } else {
    // ======================= softmax + epilogue (warps 0-3) =======================
    const int m = warp * 32 + lane;  // TMEM lane: K row (KV head m / 16, key m % 16); O^T: head dim
    const int hf = lane >> 4;        // which of the warp's two KV heads
    const int hm = 2 * warp + hf;    // this thread's KV head
    const int kk = lane & 15;        // this thread's key in the block
    const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
    float* const xch = reinterpret_cast<float*>(gb + L::OFF_XCH);
    int nx = 0;  // exchanges done; exchange x uses buffer and barrier x % 2
    constexpr float kSlack = 0.75f;  // log2 units: P' = 256 p <= 430 < 448
    constexpr float kHead = PA_TM_HEAD;  // a moved reference is set this far above the maxima
    constexpr float kHeadFirst = PA_TM_HEAD_FIRST;  // a token's first reference
    constexpr int CW = L::CW;
    // P'^T of buffer b: row r (query row; hi rows < HQ, lo rows >= HQ), byte m
    auto prow = [&](int b, int r) -> unsigned char* {
      return gb + L::OFF_P + b * L::kPBytes + r * 128 + ((((m >> 4) ^ (r & 7))) << 4) + (m & 15);
    };
    auto st_cols = [&](uint32_t taddr, const uint32_t (&v)[CW]) {
      if constexpr (CW == 16) {
        uint32_t a[8], c[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          a[j] = v[j];
          c[j] = v[8 + j];
        }
        tm_st<8>(taddr, a);
        tm_st<8>(taddr + 8, c);
      } else {
        tm_st<CW>(taddr, v);
      }
    };
    // reference max and (this thread's keys') sum of each query row of this
    // thread's KV head, in the current token
    float mr[G], lt[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      mr[g] = 0.f;
      lt[g] = 0.f;
    }
    // A token's epilogue runs during the next tile, after that tile's P is
    // released (it reads the other O^T buffer): its maxima and sums are kept.
    bool pend = false;
    int ptok = 0, pfl = 0, pi = 0;
    float pm[G], pl[G];
    auto epilogue = [&](int etok, int efl, int ei, const float (&em)[G], const float (&el)[G]) -> bool {
      // the KV heads' sums over their 16 keys, published with the maxima
      const int kx = nx++;
      float* const xb = xch + (kx & 1) * L::XCH_FLOATS;
      float sum[G];
#pragma unroll
      for (int g = 0; g < G; ++g) sum[g] = half_sum(el[g]);
      if (kk == 0) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
          xb[4 + HQ + hm * G + g] = sum[g];
          xb[4 + 2 * HQ + hm * G + g] = em[g];
        }
      }
      mbar_arrive(BAR(L::B_XCH + (kx & 1)));
      if (!wait(L::B_XCH + (kx & 1), kx >> 1)) return false;
      // the token's last P.V has completed
      if (!wait(L::B_PFREE + (ei & 1), ei >> 1)) return false;
      tc_fence_after();
      const uint32_t ob = 2u * N + ((efl & T_PAR) ? (uint32_t)N : 0u);
      const bool whole = (efl & T_WHOLE) != 0;
#pragma unroll 1
      for (int c0 = 0; c0 < HQ; c0 += CW) {
        uint32_t hi[CW], lo[CW];
        tm_ld<CW>(trow + ob + c0, hi);
        tm_ld<CW>(trow + ob + HQ + c0, lo);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < CW; ++j) {
          const int qh = c0 + j;
          const float o = (__uint_as_float(hi[j]) + __uint_as_float(lo[j])) * (1.f / 256.f);
          if (whole) {
            p.out[((size_t)etok * p.num_q_heads + qh) * kTmD + m] =
                __bfloat16_as_ushort(__float2bfloat16_rn(o * (p.v_scale / xb[4 + HQ + qh])));
          } else {
            float* const slot = p.partials + ((size_t)(etok + w) * kTmHkv + qh / G) * p.slot_floats;
            __stcg(slot + 16 + (qh % G) * kTmD + m, o);
          }
        }
      }
      if (!whole && m < HQ) {  // the partial's maxima and sums
        float* const slot = p.partials + ((size_t)(etok + w) * kTmHkv + m / G) * p.slot_floats;
        __stcg(slot + (m % G), xb[4 + 2 * HQ + m]);
        __stcg(slot + G + (m % G), xb[4 + HQ + m]);
      }
      tc_fence_before();
      return true;
    };

    int i = 0;
    bool ok = true;
#pragma unroll 1
    while (ok) {
      const int st = i % kStages;
      if (!wait(L::B_FULL + st, i / kStages)) { ok = false; break; }  // the record is visible
      const TmRec rec = recs[st];
      if (rec.flags & T_END) break;
      const int b = i & 1;  // S^T and P'^T buffer of this tile
      if (!wait(L::B_S + b, i >> 1)) { ok = false; break; }
      tc_fence_after();
      const bool valid = rec.key0 + kk < rec.len;
      // P'^T buffer b is free once the P.V of tile i - 2 has completed
      if (i >= 2 && !wait(L::B_PFREE + b, (i >> 1) - 1)) { ok = false; break; }
      // scores of this thread's key for its KV head's G query rows (hi + lo,
      // each row's 2^-e undone), in log2 units
      float t[G];
      {
        uint32_t shi[2 * G], slo[2 * G];
        const uint32_t scol = (uint32_t)(N * b + 2 * warp * G);
        tm_ld<2 * G>(trow + scol, shi);
        tm_ld<2 * G>(trow + scol + HQ, slo);
        tmem_wait_ld();
        const float* const inv =
            reinterpret_cast<const float*>(gb + L::OFF_INV + st * HQ * 4) + hm * G;
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float s = __uint_as_float(hf ? shi[G + g] : shi[g]) +
                          __uint_as_float(hf ? slo[G + g] : slo[g]);
          t[g] = valid ? s * (inv[g] * p.scale_log2) : -INFINITY;
        }
      }
      // references: the token's first tile sets them from its maxima; later
      // tiles move one only for a score above it by more than kSlack
      float alpha[G];
      bool moved = false;
#pragma unroll
      for (int g = 0; g < G; ++g) alpha[g] = 1.f;
      if (rec.flags & T_FIRST) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
          mr[g] = half_max(t[g]) + kHeadFirst;
          lt[g] = 0.f;
        }
      } else {
        bool over = false;
#pragma unroll
        for (int g = 0; g < G; ++g) over |= t[g] > mr[g] + kSlack;
        if (__any_sync(kLanes, over)) {  // warp-uniform: both halves take their maxima
#pragma unroll
          for (int g = 0; g < G; ++g) {
            const float tmx = half_max(t[g]);
            if (tmx > mr[g] + kSlack) {
              alpha[g] = exp2f(mr[g] - (tmx + kHead));
              mr[g] = tmx + kHead;
              moved = true;
            }
          }
        }
      }
      // post which heads moved (O^T columns every thread must rescale)
      const int kx = nx++;
      float* const xb = xch + (kx & 1) * L::XCH_FLOATS;
      const bool wmoved = __any_sync(kLanes, moved);
      if (kk == 0) {
#pragma unroll
        for (int g = 0; g < G; ++g) xb[4 + hm * G + g] = alpha[g];
      }
      if (lane == 0) xb[warp] = wmoved ? 1.f : 0.f;
      mbar_arrive(BAR(L::B_XCH + (kx & 1)));
      // P' = 256 p as E4M3 hi + lo on the block diagonal of P'^T
      float pr[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        pr[g] = valid ? ex2_approx(t[g] - mr[g]) : 0.f;
        lt[g] = lt[g] * alpha[g] + pr[g];
      }
#pragma unroll
      for (int g = 0; g < G; g += 2) {
        const float x0 = 256.f * pr[g], x1 = g + 1 < G ? 256.f * pr[g + 1] : 0.f;
        const uint16_t hi = float2_to_e4m3x2(x0, x1);
        const float2 hv = e4m3x2_to_float2(hi);
        const uint16_t lo = float2_to_e4m3x2(x0 - hv.x, x1 - hv.y);
        const int r = hm * G + g;
        *prow(b, r) = (unsigned char)(hi & 0xffu);
        *prow(b, HQ + r) = (unsigned char)(lo & 0xffu);
        if (g + 1 < G) {
          *prow(b, r + 1) = (unsigned char)(hi >> 8);
          *prow(b, HQ + r + 1) = (unsigned char)(lo >> 8);
        }
      }
      if (!valid) {
        // a key past the sequence end: P' = 0, but its V row may hold
        // anything (0 x NaN would poison O)
        unsigned char* const vrow =
            gb + L::OFF_STAGE + st * L::kStageBytes + L::kKvTile + m * 128;
#pragma unroll
        for (int q = 0; q < 8; ++q) *reinterpret_cast<uint4*>(vrow + q * 16) = make_uint4(0u, 0u, 0u, 0u);
      }
      fence_proxy_async_smem();  // generic-proxy stores -> visible to the tensor core
      // collect: a head that moved rescales its O^T columns before this P.V
      if (!wait(L::B_XCH + (kx & 1), kx >> 1)) { ok = false; break; }
      if ((xb[0] + xb[1]) + (xb[2] + xb[3]) != 0.f) {
        // O^T is stable once the previous tile's P.V has completed
        if (!wait(L::B_PFREE + ((i - 1) & 1), (i - 1) >> 1)) { ok = false; break; }
        tc_fence_after();
        const uint32_t ob = 2u * N + ((rec.flags & T_PAR) ? (uint32_t)N : 0u);
#pragma unroll 1
        for (int c0 = 0; c0 < HQ; c0 += CW) {
          uint32_t hi[CW], lo[CW];
          tm_ld<CW>(trow + ob + c0, hi);
          tm_ld<CW>(trow + ob + HQ + c0, lo);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < CW; ++j) {
            const float a = xb[4 + c0 + j];
            hi[j] = __float_as_uint(__uint_as_float(hi[j]) * a);
            lo[j] = __float_as_uint(__uint_as_float(lo[j]) * a);
          }
          st_cols(trow + ob + c0, hi);
          st_cols(trow + ob + HQ + c0, lo);
        }
        tmem_wait_st();
      }
      tc_fence_before();
      mbar_arrive(BAR(L::B_PREADY + b));
      if (pend) {  // the previous token's epilogue (the other O^T buffer)
        if (!epilogue(ptok, pfl, pi, pm, pl)) { ok = false; break; }
        pend = false;
      }
      if (rec.flags & T_LAST) {
        pend = true;
        ptok = rec.tok;
        pfl = rec.flags;
        pi = i;
#pragma unroll
        for (int g = 0; g < G; ++g) {
          pm[g] = mr[g];
          pl[g] = lt[g];
        }
      }
      ++i;
    }
    if (ok && pend) epilogue(ptok, pfl, pi, pm, pl);  // the last token's
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}

// ---------------------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------------------
namespace {

template <int G, int CPS>
cudaError_t launch_tm_t(const DecodeParams& d, int grid, cudaStream_t s) {
  using L = TmL<G, CPS>;
  TmDecodeParams tp;
  tp.d = d;
  const uint64_t qrows = (uint64_t)d.num_tokens * (uint64_t)d.num_q_heads;
  // q' rows as {128 B, rows (256 B apart), hi / lo (128 B apart)}: a box of a
  // token's Hq rows lands as [hi, lo][Hq rows][128 B]
  const uint64_t qd[3] = {128, qrows, 2}, qs[2] = {2 * kTmD, kTmD};
  const uint32_t qb[3] = {128, (uint32_t)L::HQ, 2};
  // a cache as {128 B, blocks * 8 * 16 rows}: a box of 128 rows is one block
  // of all eight KV heads
  const uint64_t rows = (uint64_t)d.num_blocks * kTmHkv * kBlockSize;
  const uint64_t cd[2] = {128, rows}, cs[1] = {kTmD};
  const uint32_t cb[2] = {128, (uint32_t)(kTmHkv * kBlockSize)};
  if (!encode_tmap_u8(&tp.tm_q, 3, d.qsplit, qd, qs, qb) ||
      !encode_tmap_u8(&tp.tm_k, 2, d.k_cache, cd, cs, cb) ||
      !encode_tmap_u8(&tp.tm_v, 2, d.v_cache, cd, cs, cb))
    return cudaErrorInvalidValue;
  auto kern = pa_decode_tm_kernel<G, CPS>;
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM);
    if (e != cudaSuccess) return e;
    // the whole unified on-chip memory as shared memory, so CPS CTAs fit
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kTmThreads);
  cfg.dynamicSmemBytes = L::SMEM;
  cfg.stream = s;
  // Programmatic launch after the query split (which releases its dependent
  // at its top and completes only after its own predecessor).
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tp);
}

}  // namespace

int decode_tm_workers(int group, int num_sms, int ctas_per_sm) {
  const int cps = (ctas_per_sm == 2 && group <= 4) ? 2 : 1;
  const int w = cps * num_sms;
  return w < kMaxDecodeWorkers / kTmHkv ? w : kMaxDecodeWorkers / kTmHkv;
}

bool decode_tm_supported(int head_dim, int group, int num_kv_heads, int workers) {
  return head_dim == kTmD && num_kv_heads == kTmHkv &&
         (group == 1 || group == 2 || group == 4 || group == 8) &&
         // partial slots (token + worker) * 8 + kv head fit the workspace's
         // tokens * kv heads + kMaxDecodeWorkers
         workers * kTmHkv <= kMaxDecodeWorkers;
}

cudaError_t launch_decode_tm(const DecodeParams& p, int group, int num_sms, int ctas_per_sm,
                             cudaStream_t s, int* workers_out) {
  const int grid = decode_tm_workers(group, num_sms, ctas_per_sm);
  *workers_out = grid;
  const bool two = grid > num_sms;  // two CTAs per SM
  switch (group) {
    case 1: return two ? launch_tm_t<1, 2>(p, grid, s) : launch_tm_t<1, 1>(p, grid, s);
    case 2: return two ? launch_tm_t<2, 2>(p, grid, s) : launch_tm_t<2, 1>(p, grid, s);
    case 4: return two ? launch_tm_t<4, 2>(p, grid, s) : launch_tm_t<4, 1>(p, grid, s);
    case 8: return launch_tm_t<8, 1>(p, grid, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace pa
