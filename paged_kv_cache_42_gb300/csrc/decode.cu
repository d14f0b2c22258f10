// Split-KV paged attention for one query token per work unit.
//
// What is computed ("vLLM v1 Deep Dive: How LLM(...) and the Server Boot and
// Generate", Part 3, "Step 4c - Mixed batches" and "Aside - KV cache and
// prefix caching"): for every new token of the batch, softmax attention of
// each of its query heads over the keys the token may see - all of a decode
// request's keys, or keys 0 .. ctx + j for token j of a prefill chunk on top
// of ctx cached tokens - with K/V reached through the request's block table.
// Query heads that share a KV head are processed together so each K/V block
// is read once per KV head ("vLLM: An Exhaustive Technical Study for Kernel
// Engineers", 2.4, the GQA grouping of the Triton unified attention backend).
//
// Work decomposition (ours). The planner lists every token with work and the
// number of (kv head, 16-key block) items it needs; all items of all tokens
// form one flattened sequence, token-major, then kv head, then block. The
// decode grid is persistent (a multiple of the SM count) and each warp is an
// independent worker that takes one contiguous, equally sized slice of that
// sequence, so the load balance is exact whatever the length mix. A warp
// whose slice holds a whole (token, kv head) writes the output directly;
// otherwise it writes an unnormalised partial (o, m, l) and moves on, and the
// merge pass (merge.cu), chained after this grid, combines the partials by
// log-sum-exp renormalisation ("vLLM: An Exhaustive Technical Study for
// Kernel Engineers", 2.3, cascade attention's log-sum-exp merge) in a fixed
// order (deterministic results). No warp waits on another.
//
// Data movement. Each (block, kv head) of K and of V is one contiguous
// 16 x D bf16 tile in the cache, fetched whole with a 1-D bulk async copy
// (TMA) into a per-warp ring of shared-memory stages, completion tracked by
// an mbarrier; NSTAGE-1 tiles are in flight while one is consumed. The q rows
// of a (token, kv head) ride along with its first tile. Block ids are
// prefetched 32 positions ahead with one coalesced load per warp.
//
// Arithmetic. Scores in fp32 with packed fp32x2 FMAs; q is prescaled by
// scale*log2(e) so the online softmax uses exp2. Per-token dot products are
// split over TPT lanes and reduced with a transposing butterfly of warp
// shuffles (G heads -> 1 value per lane in log2(TPT) shuffle rounds).
#include <math.h>

#include "pa_internal.h"
#include "ptx.cuh"

namespace pa {

constexpr unsigned kFull = 0xffffffffu;

// =============================================================================
// Split-KV decode kernel
// =============================================================================
// Test builds only: bytes added to every stage's expected transaction count,
// so no stage barrier ever completes and the bounded waits give up (the
// copies issued still land; see tests/test_gpu_wait_timeout.py). 0 in the
// library.
#ifndef PA_TEST_EXTRA_TX
#define PA_TEST_EXTRA_TX 0
#endif

// Largest head group whose P.V pass gives each lane 8 output dims (else 4).
// Eight dims halve the per-row overhead (address, p broadcast) of the pass at
// the price of twice the accumulator registers (measured on the Llama-8B
// decode batch: 98 us against 106 us with a bf16 cache, 106 us against
// 108 us with an E4M3 one, although its two CTAs per SM replace three).
#ifndef PA_DEC_VD8_MAXG
#define PA_DEC_VD8_MAXG 4
#endif

template <int D, int G, bool F8>
struct Cfg {
  static constexpr int EB = F8 ? 1 : 2;          // bytes per cached K/V element
  static constexpr int DPT = (G <= 4) ? 16 : 8;  // q.k dims per lane
  static constexpr int TPT = D / DPT;            // lanes per token in q.k
  static constexpr int TPP = 32 / TPT;           // tokens per q.k pass
  static constexpr int NPASS = 16 / TPP;
  static constexpr int LOG_G = G == 1 ? 0 : G == 2 ? 1 : G == 4 ? 2 : 3;
  static constexpr int VD = G <= PA_DEC_VD8_MAXG ? 8 : 4;  // output dims per lane
  static constexpr int LPR = D / VD;   // lanes per V row
  static constexpr int RPS = 32 / LPR;  // V rows per step
  static constexpr int KV_BYTES = kBlockSize * D * EB;
  static constexpr int Q_BYTES = G * D * 2;
  static constexpr int STAGE_BYTES = 2 * KV_BYTES + Q_BYTES;
  static constexpr int P_BYTES = kBlockSize * G * 4 + 64;  // p[16][G], alpha[G]
  static_assert(TPT >= G, "a token's lane group must hold one value per head");
  static_assert(DPT == 8 || DPT == 16, "one or two 16-byte chunks per lane");
  static_assert(RPS >= 1 && kBlockSize % RPS == 0, "whole V rows per step");
};

template <int D, int G, int NSTAGE, bool F8>
struct WarpSmem {
  using C = Cfg<D, G, F8>;
  static constexpr int RAW = NSTAGE * C::STAGE_BYTES + C::P_BYTES + NSTAGE * 8;
  static constexpr int BYTES = (RAW + 127) / 128 * 128;
};

// Head whose score a lane holds after the transposing reduction.
template <int G>
__device__ __forceinline__ int head_of_lane(int lane) {
  int h = 0;
#pragma unroll
  for (int st = 0; (1 << st) < G; ++st) h += ((lane >> st) & 1) * (G >> (st + 1));
  return h;
}
template <int G>
__device__ __forceinline__ int lane_of_head(int h) {
  constexpr int LOG_G = G == 1 ? 0 : G == 2 ? 1 : G == 4 ? 2 : 3;
  int lane = 0;
#pragma unroll
  for (int st = 0; st < LOG_G; ++st) lane |= ((h >> (LOG_G - 1 - st)) & 1) << st;
  return lane;
}

// Sum G per-lane partial dot products over the TPT lanes of a token group.
// Each round halves the number of live values: a lane keeps one half, sends
// the other to its partner and adds what it receives. Ends with the full sum
// for head head_of_lane<G>(lane) in every lane of the group.
template <int G, int TPT>
__device__ __forceinline__ float reduce_heads(float (&v)[G], int lane) {
#pragma unroll
  for (int st = 0; (1 << st) < TPT; ++st) {
    const int m = 1 << st;
    const int n = (G >> st) > 1 ? (G >> st) : 1;
    if (n > 1) {
      const bool upper = (lane & m) != 0;
#pragma unroll
      for (int i = 0; i < n / 2; ++i) {
        const float send = upper ? v[i] : v[i + n / 2];
        const float keep = upper ? v[i + n / 2] : v[i];
        v[i] = keep + __shfl_xor_sync(kFull, send, m);
      }
    } else {
      v[0] += __shfl_xor_sync(kFull, v[0], m);
    }
  }
  return v[0];
}

// Per-lane metadata of one position of a 32-position batch.
struct Batch {
  int k, tok, len, kv, blk, nb, pid, end;
};
struct Loc {
  int k, tok, req, len, base;
};

template <int D, int G, int WARPS, int NSTAGE, bool F8>
__device__ __forceinline__ void decode_body(const DecodeParams& p) {
  using C = Cfg<D, G, F8>;
  using WS = WarpSmem<D, G, NSTAGE, F8>;
  extern __shared__ __align__(128) unsigned char smem[];
  // The merge pass may be placed as soon as CTAs of this persistent grid
  // retire (it waits for the whole grid before reading).
  griddep_launch_dependents();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned char* const wsm = smem + warp * WS::BYTES;  // this warp's region
  const uint32_t stage0 = smem_u32(wsm);
  float* const p_s = reinterpret_cast<float*>(wsm + NSTAGE * C::STAGE_BYTES);  // [16][G]
  float* const alpha_s = reinterpret_cast<float*>(p_s + kBlockSize * G);
  const uint32_t bars = stage0 + NSTAGE * C::STAGE_BYTES + C::P_BYTES;
  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < NSTAGE; ++s) mbar_init(bars + 8 * s, 1);
    fence_barrier_init();
  }
  __syncwarp();

  // The work list: from the planner (the preceding grid), or - for a
  // decode-only batch (every span at most one token) - built by this CTA from
  // query_start_loc and seq_lens, without waiting for any earlier grid.
  const UnitInfo* units = p.units;
  int W, K;
  bool waited = false;  // lane 0: griddepcontrol.wait done (plan, KV write visible)
  if (p.self_plan) {
    UnitInfo* const su = reinterpret_cast<UnitInfo*>(smem + WARPS * WS::BYTES);
    __shared__ int s_tot[WARPS];
    const int R = p.num_reqs, T = p.num_tokens, Hkv_ = p.num_kv_heads;
    int carry = 0;
    for (int r0 = 0; r0 < R; r0 += 32 * WARPS) {
      const int r = r0 + warp * 32 + lane;
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
        const int y = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += y;
      }
      if (lane == 31) s_tot[warp] = incl;
      __syncthreads();
      int off = carry;
      for (int w2 = 0; w2 < warp; ++w2) off += s_tot[w2];
      if (r < R) su[r] = UnitInfo{q0, r, L, off + incl - n};
      for (int w2 = 0; w2 < WARPS; ++w2) carry += s_tot[w2];
      __syncthreads();
    }
    if (threadIdx.x == 0) su[R] = UnitInfo{T, -1, 0, carry};
    __syncthreads();
    if (blockIdx.x == 0 && threadIdx.x == 0) {  // the merge pass slices alike
      p.header_out->num_units = R;
      p.header_out->num_positions = carry;
    }
    units = su;
    W = carry;
    K = R;
  } else if (p.overlap) {
    // started by the cascade prefix pass once the planner (and the KV write
    // before it) had completed: the plan is read from L2, and the prefix
    // pass is waited for only at the end (see pa_decode_kernel)
    waited = true;
    W = __ldcg(&p.header->num_positions);
    K = __ldcg(&p.header->num_units);
  } else {
    griddep_wait();  // the plan is written by the preceding grid
    waited = true;
    W = p.header->num_positions;
    K = p.header->num_units;
  }
  if (W <= 0) return;
  const int launched = (int)gridDim.x * WARPS;
  const int NW = plan_workers(W, launched < p.max_workers ? launched : p.max_workers);
  const int w = blockIdx.x * WARPS + warp;
  if (w >= NW) return;
  const int S = worker_begin(w, W, NW);
  const int E = worker_begin(w + 1, W, NW);
  if (S >= E) return;
  const int Hkv = p.num_kv_heads, Hq = p.num_q_heads;
  const int kstart = p.key_start_blocks;  // first block on this path (cascade prefix skipped)


  // ---- batch metadata helpers ------------------------------------------------
  // the planner's table (global memory, an earlier grid's) is read from L2
  auto unit_at = [&](int k) -> int4 {
    return p.self_plan ? *reinterpret_cast<const int4*>(units + k)
                       : __ldcg(reinterpret_cast<const int4*>(units + k));
  };
  auto window = [&](int kbase) -> int {
    const int kk = kbase + lane;
    return kk <= K ? unit_at(kk).w : 0x7fffffff;
  };
  auto locate = [&](int y0, int kbase, int win) -> Loc {
    const int y = y0 + lane;
    int c = 0;
#pragma unroll
    for (int i = 0; i < 32; ++i) c += (__shfl_sync(kFull, win, i) <= y) ? 1 : 0;
    int k = kbase + c - 1;
    k = k < 0 ? 0 : (k > K ? K : k);
    const int4 u = unit_at(k);
    return Loc{k, u.x, u.y, u.z, u.w};
  };
  auto finish = [&](int y0, const Loc& kl) -> Batch {
    Batch b;
    const int y = y0 + lane;
    b.k = kl.k;
    b.tok = kl.tok;
    b.len = kl.len;
    const int base = kl.base;
    int nb = (b.len + kBlockSize - 1) / kBlockSize - kstart;  // blocks after a cascade prefix
    nb = nb < 1 ? 1 : nb;
    b.nb = nb;
    b.end = base + nb * Hkv;
    const int off = y - base;
    b.kv = off / nb;
    b.blk = off - b.kv * nb;
    int pid = 0;
    if (y < E) {
      pid = __ldg(p.block_tables + (size_t)kl.req * p.bt_stride + kstart + b.blk);
      if (pid < 0 || pid >= p.num_blocks) {
        report_error(p.err, PA_DEVERR_BLOCK_ID, y);
        pid = 0;
      }
    }
    b.pid = pid;
    return b;
  };

  // ---- the unit holding the first position: from the planner, or a 32-ary
  // search over units[].base --------------------------------------------------------
  int lo = 0, hi = K;  // base[lo] <= S < base[hi]
  if (p.worker_unit && !p.self_plan) {
    lo = __ldcg(p.worker_unit + w);
    hi = lo + 1;
  }
#pragma unroll 1
  while (hi - lo > 1) {
    const int step = (hi - lo + 31) / 32;
    const int idx = lo + lane * step;
    const bool ok = idx < hi && unit_at(idx).w <= S;
    const unsigned bal = __ballot_sync(kFull, ok);
    const int last = 31 - __clz(bal);
    lo = lo + last * step;
    hi = min(hi, lo + step);
  }

  Batch cur = finish(S, locate(S, lo, window(lo)));
  Batch nxt = cur;
  if (w > 0) {  // the merge task of the slice boundary before this worker
    const int tok0 = __shfl_sync(kFull, cur.tok, 0), kv0 = __shfl_sync(kFull, cur.kv, 0);
    const int blk0 = __shfl_sync(kFull, cur.blk, 0), nb0 = __shfl_sync(kFull, cur.nb, 0);
    if (lane == 0) {
      int4 task = make_int4(-1, 0, 0, 0);
      if (blk0 != 0) {  // the slice starts inside a (token, kv head)
        const int first = S - blk0;
        const int wf = worker_of(first, W, NW);
        if (w == wf + 1) task = make_int4(tok0, kv0, wf, worker_of(first + nb0 - 1, W, NW));
      }
      p.merge_tasks[w] = task;
    }
  }
  int y0 = S;
  int nwin = 0, nkbase = 0;
  Loc nkl{0, 0, 0, 0, 0};

  // last: the segment's last block, which holds the new token of a decode; in a
  // self-planned launch its K/V come from the KV write, so wait for it first.
  auto issue = [&](int stage, int pid, int kv, bool with_q, int tok, bool last) {
    if (lane == 0) {
      if (last && !waited) {
        griddep_wait();
        waited = true;
      }
      const uint32_t dst = stage0 + stage * C::STAGE_BYTES;
      const uint32_t bar = bars + 8 * stage;
      const size_t off = ((size_t)pid * Hkv + kv) * (kBlockSize * D) * C::EB;  // bytes
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(bar, 2 * C::KV_BYTES + (with_q ? C::Q_BYTES : 0) + PA_TEST_EXTRA_TX);
      bulk_g2s(dst, static_cast<const unsigned char*>(p.k_cache) + off, C::KV_BYTES, bar);
      bulk_g2s(dst + C::KV_BYTES, static_cast<const unsigned char*>(p.v_cache) + off, C::KV_BYTES,
               bar);
      if (with_q)
        bulk_g2s(dst + 2 * C::KV_BYTES, p.q + ((size_t)tok * Hq + (size_t)kv * G) * D, C::Q_BYTES,
                 bar);
    }
  };

  // prologue
#pragma unroll
  for (int i = 0; i < NSTAGE; ++i) {
    if (S + i < E) {
      const int pid = __shfl_sync(kFull, cur.pid, i);
      const int kv = __shfl_sync(kFull, cur.kv, i);
      const int blk = __shfl_sync(kFull, cur.blk, i);
      const int tok = __shfl_sync(kFull, cur.tok, i);
      const int nbi = __shfl_sync(kFull, cur.nb, i);
      issue(i, pid, kv, i == 0 || blk == 0, tok, blk == nbi - 1);
    }
  }

  // ---- per-lane roles ---------------------------------------------------------------
  const int sub = lane % C::TPT;                                 // q.k dim slice
  const int tg = lane / C::TPT;                                  // token within a pass
  // bf16 rows: a lane's 32 bytes are two 16-byte chunks, read in an order
  // that avoids bank conflicts; E4M3 rows: one chunk, natural order
  const int swz = (!F8 && C::DPT == 16) ? ((lane >> 2) & 1) : 0;
  const int hsel = head_of_lane<G>(lane);
  const int rl = lane % C::LPR;                                  // V dims VD*rl .. VD*rl+VD-1
  const int rrow = lane / C::LPR;                                // V row within a step

  float2 qv[G][C::DPT / 2];
  float2 acc[G][C::VD / 2];
  float m_run = -INFINITY, l_run = 0.f;
#pragma unroll
  for (int h = 0; h < G; ++h) {
#pragma unroll
    for (int i = 0; i < C::VD / 2; ++i) acc[h][i] = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < C::DPT / 2; ++i) qv[h][i] = make_float2(0.f, 0.f);
  }

  int stage = 0;
  uint32_t phase = 0;
#pragma unroll 1
  for (int y = S; y < E; ++y) {
    int j = y - y0;
    if (j == 32) {
      cur = nxt;
      y0 += 32;
      j = 0;
    }
    if (y0 + 32 < E) {  // stage the metadata of the next batch, a step at a time
      if (j == 0) {
        const int k31 = __shfl_sync(kFull, cur.k, 31);
        const int end31 = __shfl_sync(kFull, cur.end, 31);
        nkbase = (y0 + 32 >= end31) ? k31 + 1 : k31;
        nwin = window(nkbase);
      } else if (j == 8) {
        nkl = locate(y0 + 32, nkbase, nwin);
      } else if (j == 16) {
        nxt = finish(y0 + 32, nkl);
      }
    }
    const int kk = __shfl_sync(kFull, cur.k, j);
    const int tok = __shfl_sync(kFull, cur.tok, j);
    const int len = __shfl_sync(kFull, cur.len, j);
    const int kv = __shfl_sync(kFull, cur.kv, j);
    const int blk = __shfl_sync(kFull, cur.blk, j);
    const int nb = __shfl_sync(kFull, cur.nb, j);
    const bool seg_start = (y == S) || blk == 0;
    const bool seg_end = (y == E - 1) || blk == nb - 1;
    const unsigned char* const st_ptr = wsm + stage * C::STAGE_BYTES;
    const uint32_t bar = bars + 8 * stage;

    if (!mbar_wait_bounded(bar, phase)) {
      if (lane == 0) report_error(p.err, PA_DEVERR_WAIT_TIMEOUT, y);
      // let every copy still in flight land before the CTA can exit
      int st2 = stage;
      uint32_t ph2 = phase;
      for (int y2 = y; y2 < E && y2 < y + NSTAGE; ++y2) {
        mbar_wait_bounded(bars + 8 * st2, ph2);
        if (++st2 == NSTAGE) { st2 = 0; ph2 ^= 1; }
      }
      return;
    }

    if (seg_start) {
      const unsigned char* const qbase = st_ptr + 2 * C::KV_BYTES;
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const unsigned char* const row = qbase + h * D * 2 + sub * C::DPT * 2;
        const uint4 a = *reinterpret_cast<const uint4*>(row + 16 * swz);
        qv[h][0] = bf16x2_to_float2(a.x);
        qv[h][1] = bf16x2_to_float2(a.y);
        qv[h][2] = bf16x2_to_float2(a.z);
        qv[h][3] = bf16x2_to_float2(a.w);
        if constexpr (C::DPT == 16) {
          const uint4 b = *reinterpret_cast<const uint4*>(row + 16 * (1 - swz));
          qv[h][4] = bf16x2_to_float2(b.x);
          qv[h][5] = bf16x2_to_float2(b.y);
          qv[h][6] = bf16x2_to_float2(b.z);
          qv[h][7] = bf16x2_to_float2(b.w);
        }
#pragma unroll
        for (int i = 0; i < C::DPT / 2; ++i)
          qv[h][i] = fmul2(qv[h][i], make_float2(p.scale_log2, p.scale_log2));
#pragma unroll
        for (int i = 0; i < C::VD / 2; ++i) acc[h][i] = make_float2(0.f, 0.f);
      }
      m_run = -INFINITY;
      l_run = 0.f;
    }

    const int nvalid = min(kBlockSize, len - (kstart + blk) * kBlockSize);

    // ---- scores: s = (q * scale * log2 e) . k for the lane's (head, token) ---------
    float sc[C::NPASS];
#pragma unroll
    for (int ps = 0; ps < C::NPASS; ++ps) {
      const int t = ps * C::TPP + tg;
      const unsigned char* const row = st_ptr + t * D * C::EB + sub * C::DPT * C::EB;
      float2 kf[C::DPT / 2];
      if constexpr (F8) {  // E4M3 codes, dequantised exactly (k_scale is folded into q)
        if constexpr (C::DPT == 16) {
          const uint4 a = *reinterpret_cast<const uint4*>(row);
          const uint32_t wv[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            kf[2 * i] = e4m3x2_to_float2((uint16_t)(wv[i] & 0xffffu));
            kf[2 * i + 1] = e4m3x2_to_float2((uint16_t)(wv[i] >> 16));
          }
        } else {
          const uint2 a = *reinterpret_cast<const uint2*>(row);
          kf[0] = e4m3x2_to_float2((uint16_t)(a.x & 0xffffu));
          kf[1] = e4m3x2_to_float2((uint16_t)(a.x >> 16));
          kf[2] = e4m3x2_to_float2((uint16_t)(a.y & 0xffffu));
          kf[3] = e4m3x2_to_float2((uint16_t)(a.y >> 16));
        }
      } else {
        const uint4 a = *reinterpret_cast<const uint4*>(row + 16 * swz);
        kf[0] = bf16x2_to_float2(a.x);
        kf[1] = bf16x2_to_float2(a.y);
        kf[2] = bf16x2_to_float2(a.z);
        kf[3] = bf16x2_to_float2(a.w);
        if constexpr (C::DPT == 16) {
          const uint4 b = *reinterpret_cast<const uint4*>(row + 16 * (1 - swz));
          kf[4] = bf16x2_to_float2(b.x);
          kf[5] = bf16x2_to_float2(b.y);
          kf[6] = bf16x2_to_float2(b.z);
          kf[7] = bf16x2_to_float2(b.w);
        }
      }
      float part[G];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float2 a2 = fmul2(qv[h][0], kf[0]);
#pragma unroll
        for (int i = 1; i < C::DPT / 2; ++i) a2 = ffma2(qv[h][i], kf[i], a2);
        part[h] = a2.x + a2.y;
      }
      sc[ps] = reduce_heads<G, C::TPT>(part, lane);
    }
    if (nvalid < kBlockSize) {  // keys past the sequence end (their slots may hold anything)
#pragma unroll
      for (int ps = 0; ps < C::NPASS; ++ps)
        if (ps * C::TPP + tg >= nvalid) sc[ps] = -INFINITY;
    }

    // ---- online softmax (base 2) ------------------------------------------------------
    float mb = sc[0];
#pragma unroll
    for (int ps = 1; ps < C::NPASS; ++ps) mb = fmaxf(mb, sc[ps]);
#pragma unroll
    for (int o = C::TPT; o < 32; o <<= 1) mb = fmaxf(mb, __shfl_xor_sync(kFull, mb, o));
    const float m_new = fmaxf(m_run, mb);
    const float alpha = exp2f(m_run - m_new);
    float psum = 0.f;
#pragma unroll
    for (int ps = 0; ps < C::NPASS; ++ps) {
      const float pr = exp2f(sc[ps] - m_new);
      psum += pr;
      p_s[(ps * C::TPP + tg) * G + hsel] = pr;
    }
    l_run = l_run * alpha + psum;
    m_run = m_new;
    // The accumulators need rescaling only when some head's running max moved
    // (and not at all right after a segment start, when they are zero).
    const bool rescale = !seg_start && !__all_sync(kFull, alpha == 1.f);
    if (rescale && lane < G) alpha_s[hsel] = alpha;
    __syncwarp();

    // ---- o = o * alpha + sum_t p_t v_t ---------------------------------------------------
    {
      if (rescale) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float al = alpha_s[h];
#pragma unroll
          for (int i = 0; i < C::VD / 2; ++i) acc[h][i] = fmul2(acc[h][i], make_float2(al, al));
        }
      }
      // Keys past the sequence end have p = 0; their V rows (which may hold
      // anything, NaN included) are replaced by the last valid row so the
      // loop needs no per-token branch: 0 * finite adds nothing.
      const unsigned char* const vbase = st_ptr + C::KV_BYTES + rl * C::VD * C::EB;
      const int tmax = nvalid - 1;
#pragma unroll
      for (int stp = 0; stp < kBlockSize / C::RPS; ++stp) {
        const int t = stp * C::RPS + rrow;
        {
          float2 vf[C::VD / 2];
          const unsigned char* const vrow = vbase + min(t, tmax) * D * C::EB;
          if constexpr (F8) {  // v_scale is applied to the output
            if constexpr (C::VD == 8) {
              const uint2 vv = *reinterpret_cast<const uint2*>(vrow);
              vf[0] = e4m3x2_to_float2((uint16_t)(vv.x & 0xffffu));
              vf[1] = e4m3x2_to_float2((uint16_t)(vv.x >> 16));
              vf[2] = e4m3x2_to_float2((uint16_t)(vv.y & 0xffffu));
              vf[3] = e4m3x2_to_float2((uint16_t)(vv.y >> 16));
            } else {
              const uint32_t vv = *reinterpret_cast<const uint32_t*>(vrow);
              vf[0] = e4m3x2_to_float2((uint16_t)(vv & 0xffffu));
              vf[1] = e4m3x2_to_float2((uint16_t)(vv >> 16));
            }
          } else if constexpr (C::VD == 8) {
            const uint4 vv = *reinterpret_cast<const uint4*>(vrow);
            vf[0] = bf16x2_to_float2(vv.x);
            vf[1] = bf16x2_to_float2(vv.y);
            vf[2] = bf16x2_to_float2(vv.z);
            vf[3] = bf16x2_to_float2(vv.w);
          } else {
            const uint2 vv = *reinterpret_cast<const uint2*>(vrow);
            vf[0] = bf16x2_to_float2(vv.x);
            vf[1] = bf16x2_to_float2(vv.y);
          }
          float2 ph[G];
          if constexpr (G >= 4) {
#pragma unroll
            for (int h4 = 0; h4 < G; h4 += 4) {
              const float4 q4 = *reinterpret_cast<const float4*>(p_s + t * G + h4);
              ph[h4] = make_float2(q4.x, q4.x);
              ph[h4 + 1] = make_float2(q4.y, q4.y);
              ph[h4 + 2] = make_float2(q4.z, q4.z);
              ph[h4 + 3] = make_float2(q4.w, q4.w);
            }
          } else if constexpr (G == 2) {
            const float2 q2 = *reinterpret_cast<const float2*>(p_s + t * 2);
            ph[0] = make_float2(q2.x, q2.x);
            ph[1] = make_float2(q2.y, q2.y);
          } else {
            ph[0] = make_float2(p_s[t], p_s[t]);
          }
#pragma unroll
          for (int h = 0; h < G; ++h) {
#pragma unroll
            for (int i = 0; i < C::VD / 2; ++i) acc[h][i] = ffma2(ph[h], vf[i], acc[h][i]);
          }
        }
      }
    }
    __syncwarp();  // every lane is done with this stage and with p_s

    // ---- refill this stage with the position NSTAGE ahead -----------------------------------
    {
      const int yi = y + NSTAGE;
      if (yi < E) {
        const int ji = yi - y0;
        int pid, kvi, blki, toki, nbi;
        if (ji < 32) {
          pid = __shfl_sync(kFull, cur.pid, ji);
          kvi = __shfl_sync(kFull, cur.kv, ji);
          blki = __shfl_sync(kFull, cur.blk, ji);
          toki = __shfl_sync(kFull, cur.tok, ji);
          nbi = __shfl_sync(kFull, cur.nb, ji);
        } else {
          pid = __shfl_sync(kFull, nxt.pid, ji - 32);
          kvi = __shfl_sync(kFull, nxt.kv, ji - 32);
          blki = __shfl_sync(kFull, nxt.blk, ji - 32);
          toki = __shfl_sync(kFull, nxt.tok, ji - 32);
          nbi = __shfl_sync(kFull, nxt.nb, ji - 32);
        }
        issue(stage, pid, kvi, blki == 0, toki, blki == nbi - 1);
      }
    }
    if (++stage == NSTAGE) {
      stage = 0;
      phase ^= 1;
    }

    if (seg_end) {
      // complete row sums and gather (m, l) of every head into every lane
      float lsum = l_run;
#pragma unroll
      for (int o = C::TPT; o < 32; o <<= 1) lsum += __shfl_xor_sync(kFull, lsum, o);
      float mh[G], lh[G];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const int src = lane_of_head<G>(h);
        mh[h] = __shfl_sync(kFull, m_run, src);
        lh[h] = __shfl_sync(kFull, lsum, src);
      }
      // the RPS row groups of the P.V pass each hold part of every output dim
#pragma unroll
      for (int o = C::LPR; o < 32; o <<= 1) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
#pragma unroll
          for (int i = 0; i < C::VD / 2; ++i) {
            acc[h][i].x += __shfl_xor_sync(kFull, acc[h][i].x, o);
            acc[h][i].y += __shfl_xor_sync(kFull, acc[h][i].y, o);
          }
        }
      }
      const int ustart = y - blk;  // first position of this (token, kv head)
      const int wf = worker_of(ustart, W, NW), wl = worker_of(ustart + nb - 1, W, NW);
      uint16_t* orow = p.out + ((size_t)tok * Hq + (size_t)kv * G) * D + rl * C::VD;
      // the lane's VD output dims of head h, scaled by f, as bf16
      auto store_out = [&](int h, const float* o, float f) {
        if constexpr (C::VD == 8) {
          uint4 pk;
          pk.x = float2_to_bf16x2(o[0] * f, o[1] * f);
          pk.y = float2_to_bf16x2(o[2] * f, o[3] * f);
          pk.z = float2_to_bf16x2(o[4] * f, o[5] * f);
          pk.w = float2_to_bf16x2(o[6] * f, o[7] * f);
          *reinterpret_cast<uint4*>(orow + h * D) = pk;
        } else {
          uint2 pk;
          pk.x = float2_to_bf16x2(o[0] * f, o[1] * f);
          pk.y = float2_to_bf16x2(o[2] * f, o[3] * f);
          *reinterpret_cast<uint2*>(orow + h * D) = pk;
        }
      };
      // Cascade: the prefix partials of this (token, kv head), one per key
      // chunk, folded into (M, Ls, O) by log-sum-exp renormalisation.
      auto fold_prefix = [&](float (&M)[G], float (&Ls)[G], float (&O)[G][C::VD]) {
#pragma unroll 1
        for (int c = 0; c < p.prefix_chunks; ++c) {
          const float* sl =
              p.prefix_partials + ((size_t)c * p.num_tokens + tok) * Hkv * p.slot_floats +
              (size_t)kv * p.slot_floats;
#pragma unroll
          for (int h = 0; h < G; ++h) {
            const float ms = __ldcg(sl + h);
            const float mn = fmaxf(M[h], ms);
            const float a = exp2f(M[h] - mn), b = exp2f(ms - mn);
            Ls[h] = Ls[h] * a + __ldcg(sl + G + h) * b;
#pragma unroll
            for (int i = 0; i < C::VD / 4; ++i) {
              const float4 o =
                  __ldcg(reinterpret_cast<const float4*>(sl + 16 + h * D + rl * C::VD) + i);
              O[h][4 * i] = O[h][4 * i] * a + o.x * b;
              O[h][4 * i + 1] = O[h][4 * i + 1] * a + o.y * b;
              O[h][4 * i + 2] = O[h][4 * i + 2] * a + o.z * b;
              O[h][4 * i + 3] = O[h][4 * i + 3] * a + o.w * b;
            }
            M[h] = mn;
          }
        }
      };
      if (wf == wl && !p.fold_later) {
        if (p.prefix_partials) {
          float M[G], Ls[G], O[G][C::VD];
#pragma unroll
          for (int h = 0; h < G; ++h) {
            M[h] = mh[h];
            Ls[h] = lh[h];
#pragma unroll
            for (int i = 0; i < C::VD / 2; ++i) {
              O[h][2 * i] = acc[h][i].x;
              O[h][2 * i + 1] = acc[h][i].y;
            }
          }
          fold_prefix(M, Ls, O);
          if (rrow == 0) {
#pragma unroll
            for (int h = 0; h < G; ++h) store_out(h, O[h], p.v_scale / Ls[h]);
          }
        } else if (rrow == 0) {
#pragma unroll
          for (int h = 0; h < G; ++h) {
            float o[C::VD];
#pragma unroll
            for (int i = 0; i < C::VD / 2; ++i) {
              o[2 * i] = acc[h][i].x;
              o[2 * i + 1] = acc[h][i].y;
            }
            store_out(h, o, p.v_scale / lh[h]);
          }
        }
      } else {
        // a partial (m, l, o) for the merge pass, in slot u + w: tokens
        // increase with the position order, so the slot is unique per segment
        const int u = tok * Hkv + kv;
        float* slot = p.partials + (size_t)(u + w) * p.slot_floats;
        if (lane == 0) {
#pragma unroll
          for (int h = 0; h < G; ++h) {
            __stcg(slot + h, mh[h]);
            __stcg(slot + G + h, lh[h]);
          }
        }
        if (rrow == 0) {
#pragma unroll
          for (int h = 0; h < G; ++h) {
#pragma unroll
            for (int i = 0; i < C::VD / 4; ++i)
              __stcg(reinterpret_cast<float4*>(slot + 16 + h * D + rl * C::VD) + i,
                     make_float4(acc[h][2 * i].x, acc[h][2 * i].y, acc[h][2 * i + 1].x,
                                 acc[h][2 * i + 1].y));
          }
        }
      }
    }
  }
}

template <int D, int G, int WARPS, int NSTAGE, bool F8>
__global__ void __launch_bounds__(WARPS * 32) pa_decode_kernel(const DecodeParams p) {
  decode_body<D, G, WARPS, NSTAGE, F8>(p);
  // overlapped cascade: complete only after the prefix pass's grid, so that
  // the merge pass after this grid sees the prefix partials too
  if (p.overlap && threadIdx.x == 0) griddep_wait();
}

// ---- launch ---------------------------------------------------------------------------

// Grid of a split-KV launch on the current device: every SM filled to its
// occupancy, capped so the workers fit the workspace's partial slots.
// Dynamic shared memory of a launch: the warps' rings, plus the unit table of
// a self-planned launch.
template <int D, int G, int WARPS, int NSTAGE, bool F8>
constexpr int decode_smem(bool self_plan) {
  return WARPS * WarpSmem<D, G, NSTAGE, F8>::BYTES +
         (self_plan ? (int)sizeof(UnitInfo) * (kSelfPlanMaxReqs + 1) : 0);
}

template <int D, int G, int WARPS, int NSTAGE, bool F8>
cudaError_t decode_grid(int num_sms, int occ_cap, bool self_plan, int* grid_out) {
  auto kern = pa_decode_kernel<D, G, WARPS, NSTAGE, F8>;
  const int smem = decode_smem<D, G, WARPS, NSTAGE, F8>(self_plan);
  static int occ_cache[64][2] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int occ = (dev >= 0 && dev < 64) ? occ_cache[dev][self_plan] : 0;
  if (occ == 0) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             decode_smem<D, G, WARPS, NSTAGE, F8>(true));
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, WARPS * 32, smem);
    if (e != cudaSuccess) return e;
    if (occ < 1) occ = 1;
    if (dev >= 0 && dev < 64) occ_cache[dev][self_plan] = occ;
  }
  if (occ > occ_cap) occ = occ_cap;
  int grid = num_sms * occ;
  if (grid * WARPS > kMaxDecodeWorkers) grid = kMaxDecodeWorkers / WARPS;
  *grid_out = grid;
  return cudaSuccess;
}

template <int D, int G, int WARPS, int NSTAGE, bool F8>
cudaError_t launch_decode_t(const DecodeParams& p, int num_sms, int occ_cap, cudaStream_t s,
                            int* workers_out) {
  auto kern = pa_decode_kernel<D, G, WARPS, NSTAGE, F8>;
  const int smem = decode_smem<D, G, WARPS, NSTAGE, F8>(p.self_plan != 0);
  int grid = 0;
  cudaError_t e = decode_grid<D, G, WARPS, NSTAGE, F8>(num_sms, occ_cap, p.self_plan != 0, &grid);
  if (e != cudaSuccess) return e;
  *workers_out = grid * WARPS;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(WARPS * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  // Programmatic launch: the grid starts when the preceding grid triggers
  // (the KV write at its top for a self-planned batch, which has no planner;
  // otherwise the planner or the tensor-core grid, at their end).
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

// Warps per CTA and ring stages per warp. Each warp owns its ring, so these
// set how many (block, kv head) tiles are in flight per SM and how many warps
// hide each other's latency; shared memory per SM is the budget they share.
#ifndef PA_DEC128_WARPS
#define PA_DEC128_WARPS 4
#endif
#ifndef PA_DEC128_STAGES
#define PA_DEC128_STAGES 2
#endif
#ifndef PA_DEC128G8_WARPS
#define PA_DEC128G8_WARPS 4
#endif
#ifndef PA_DEC128G8_STAGES
#define PA_DEC128G8_STAGES 2
#endif
#ifndef PA_DEC64_WARPS
#define PA_DEC64_WARPS 4
#endif
#ifndef PA_DEC64_STAGES
#define PA_DEC64_STAGES 3
#endif

#ifndef PA_DEC128F8_STAGES
#define PA_DEC128F8_STAGES 3
#endif
#ifndef PA_DEC64F8_STAGES
#define PA_DEC64F8_STAGES 3
#endif

// Warps per CTA and ring stages per warp of each instantiation. An E4M3 tile
// is half the bytes of a bf16 one: three-stage FP8 rings still leave room for
// a third CTA per SM where registers allow it (groups of up to two heads).
template <int D, int G, bool F8>
struct Tuning {
  static constexpr int WARPS =
      D == 128 ? (G == 8 ? PA_DEC128G8_WARPS : PA_DEC128_WARPS) : PA_DEC64_WARPS;
  static constexpr int STAGES =
      F8 ? (D == 128 ? PA_DEC128F8_STAGES : PA_DEC64F8_STAGES)
         : (D == 128 ? (G == 8 ? PA_DEC128G8_STAGES : PA_DEC128_STAGES) : PA_DEC64_STAGES);
};

template <int D, int G, bool F8>
cudaError_t launch_one(const DecodeParams& p, int num_sms, int occ_cap, cudaStream_t s,
                       int* workers_out) {
  using T = Tuning<D, G, F8>;
  return launch_decode_t<D, G, T::WARPS, T::STAGES, F8>(p, num_sms, occ_cap, s, workers_out);
}

template <int D, int G, bool F8>
int workers_one(int num_sms, int occ_cap) {
  using T = Tuning<D, G, F8>;
  int grid = 0;
  if (decode_grid<D, G, T::WARPS, T::STAGES, F8>(num_sms, occ_cap, false, &grid) != cudaSuccess)
    return 0;
  return grid * T::WARPS;
}

// Calls FN<D, G, F8>(args...) for the runtime (head_dim, group, f8).
#define PA_DECODE_DISPATCH(FN, FAIL, ...)                                             \
  do {                                                                                \
    if (head_dim == 128) {                                                            \
      switch (group) {                                                                \
        case 1: return f8 ? FN<128, 1, true>(__VA_ARGS__) : FN<128, 1, false>(__VA_ARGS__); \
        case 2: return f8 ? FN<128, 2, true>(__VA_ARGS__) : FN<128, 2, false>(__VA_ARGS__); \
        case 4: return f8 ? FN<128, 4, true>(__VA_ARGS__) : FN<128, 4, false>(__VA_ARGS__); \
        case 8: return f8 ? FN<128, 8, true>(__VA_ARGS__) : FN<128, 8, false>(__VA_ARGS__); \
      }                                                                               \
    } else if (head_dim == 64) {                                                      \
      switch (group) {                                                                \
        case 1: return f8 ? FN<64, 1, true>(__VA_ARGS__) : FN<64, 1, false>(__VA_ARGS__);   \
        case 2: return f8 ? FN<64, 2, true>(__VA_ARGS__) : FN<64, 2, false>(__VA_ARGS__);   \
        case 4: return f8 ? FN<64, 4, true>(__VA_ARGS__) : FN<64, 4, false>(__VA_ARGS__);   \
        case 8: return f8 ? FN<64, 8, true>(__VA_ARGS__) : FN<64, 8, false>(__VA_ARGS__);   \
      }                                                                               \
    }                                                                                 \
    return FAIL;                                                                      \
  } while (0)

cudaError_t launch_decode(const DecodeParams& p, int head_dim, int group, bool f8, int num_sms,
                          int occ_cap, cudaStream_t s, int* workers_out) {
  PA_DECODE_DISPATCH(launch_one, cudaErrorInvalidValue, p, num_sms, occ_cap, s, workers_out);
}

int decode_workers(int head_dim, int group, bool f8, int num_sms, int occ_cap) {
  PA_DECODE_DISPATCH(workers_one, 0, num_sms, occ_cap);
}

}  // namespace pa
