// Prefill-chunk attention on the tensor cores (tcgen05 + TMEM + TMA).
//
// What is computed ("vLLM v1 Deep Dive: How LLM(...) and the Server Boot and
// Generate", Part 3, "Aside - KV cache and prefix caching": a prefill query
// attends causally over [its already-cached prefix blocks] + [its new
// tokens]): for a request with ctx cached tokens and a chunk of qlen new
// tokens, new token j attends to keys 0 .. ctx + j, K/V read through the
// request's block table.
//
// Tiling (ours). A row tile is 128 query rows of one (request, kv head): the G
// query heads of the kv head times 128/G consecutive chunk tokens, row
// m = token * G + head - the GQA "Q block" packing ("vLLM: An Exhaustive
// Technical Study for Kernel Engineers", 2.4, Triton unified attention), so a
// row tile shares one K/V stream. A CTA work item is a PAIR of adjacent row
// tiles (256 rows) over the same keys; keys come in tiles of 128 = eight
// 16-key cache blocks, loaded once for both row tiles.
//
//   S_t = Q_t K^T   tcgen05.mma kind::f16, M=128 N=128, A=Q_t and B=K from
//                   128B-swizzled shared memory, fp32 into TMEM.
//   softmax         one thread per row (one TMEM lane): mask, scale, running
//                   max, exp2; P_t rounded to bf16 and written back into TMEM
//                   over the S_t it came from.
//   O_t += P_t V    tcgen05.mma with A=P_t from TMEM, B=V (M/N-major) from
//                   shared memory, O_t in TMEM.
// The two row tiles ping-pong: while one warpgroup runs the softmax of its
// tile, the tensor core runs the other tile's P*V and next S.
//
// The running max is only moved (and O rescaled through TMEM) when it grows
// by more than 2^8; otherwise P is formed against the stale max, which keeps
// every P <= 256 and the result exact up to rounding.
//
// Cascade prefix pass (the PREFIX instantiation; "vLLM: An Exhaustive
// Technical Study for Kernel Engineers", 2.3, cascade attention): the same
// pipeline over the common prefix shared by every request of the batch. A
// work item is (pair of row tiles of consecutive batch tokens, kv head, chunk
// of prefix key tiles); every row sees every prefix key (the prefix lies in
// each request's context), and the epilogue writes an fp32 partial (running
// max, sum, unnormalised output) per (chunk, token, kv head) for the split-KV
// kernel to merge, instead of bf16 rows.
//
// FP8 caches (the F8 instantiation; "vLLM: An Exhaustive Technical Study for
// Kernel Engineers", 2.8: E4M3 codes with per-tensor k_scale / v_scale): four
// more warps (448 threads) load each key tile's E4M3 rows with plain
// coalesced loads (one thread per key row) and widen them to bf16 - exactly,
// every E4M3 value being a bf16 - straight into the 128B-swizzled operand
// layout the MMA reads, then arrive on the stage's full barrier. k_scale is
// folded into the softmax scale and v_scale into the epilogue.
//
// Warp roles (320 threads): warp 0 issues TMA loads (both Q tiles per work
// item, K into a 3-stage ring released right after both S MMAs of a key tile,
// V into a 2-stage ring released after both P*V), warp 1 allocates TMEM and
// one thread issues the MMAs in order
//   S0(0) S1(0) | PV0(i) S0(i+1) PV1(i) S1(i+1) | ...
// and warps 2-5 / 6-9 (warpgroup t; warp w reads TMEM lanes 32*(w%4)..) run
// the softmax and epilogue of row tile t. Every wait is bounded; a wait that
// gives up sets the device error word and the CTA winds down.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "pa_internal.h"
#include "ptx.cuh"

namespace pa {

namespace {

constexpr unsigned kAll = 0xffffffffu;

// Threads per S row in the softmax (1 or 2). With 2, the two threads of a row
// take 64 score columns each and combine their row maxima through shared
// memory (a bounded mbarrier exchange). It shortens the softmax but not the
// kernel: in steady state the tensor pipe, not the softmax, sets the pace of
// a key tile (measured 52.6 us with 2 vs 51.4 us with 1 on the mixed batch),
// so the default is 1.
#ifndef PA_PREFILL_SPLIT
#define PA_PREFILL_SPLIT 1
#endif
constexpr int kSplit = PA_PREFILL_SPLIT;
static_assert(kSplit == 1 || kSplit == 2, "one or two threads per row");

template <int D, int G>
struct PCfg {
  static constexpr int TOK = 128 / G;         // chunk tokens per 128-row tile
  static constexpr int NCH = D / 64;          // 64-element (128-byte) d chunks
  static constexpr int CHUNK = 128 * 128;     // one [128 rows][128 B] operand chunk
  static constexpr int Q_BYTES = NCH * CHUNK; // one row tile of Q
  static constexpr int KV_BYTES = NCH * CHUNK;  // one 128-key tile of K or of V
  // a third K stage does not fit beside the row-max exchange buffer
#ifdef PA_PREFILL_KSTAGES
  static constexpr int KSTAGES = PA_PREFILL_KSTAGES;
#else
  static constexpr int KSTAGES = kSplit == 2 ? 2 : 3;
#endif
  static constexpr int VSTAGES = 2;
  static constexpr int OFF_Q = 0;  // two row tiles
  static constexpr int OFF_K = OFF_Q + 2 * Q_BYTES;
  static constexpr int OFF_V = OFF_K + KSTAGES * KV_BYTES;
  static constexpr int OFF_BAR = OFF_V + VSTAGES * KV_BYTES;
  // row-max / row-sum exchange of the split softmax: [row tile][parity][half][128 rows]
  static constexpr int OFF_XCH = OFF_BAR + 256;
  static constexpr int XCH_BYTES = kSplit == 2 ? 2 * 2 * 2 * 128 * 4 : 0;
  static constexpr int SMEM = OFF_XCH + XCH_BYTES + 1024;  // + 1 KB alignment slack
  static constexpr uint32_t TMEM_COLS = 512;
  // S_t (fp32, 128 columns) at 128*t; P_t (bf16 pairs, 64 columns) is written
  // over S_t, each thread's part over its own S columns (P column of key k:
  // pcol(k / 32) + (k % 32) / 2); O_t at 256 + 128*t.
  static constexpr uint32_t TM_S = 0;
  static constexpr uint32_t TM_O = 256;
  static constexpr int CPH = 4 / kSplit;  // 32-column S chunks per softmax thread
  // first P column of S chunk c: chunk c's 32 scores become 16 bf16 pairs
  __host__ __device__ static constexpr uint32_t pcol(int c) {
    return 64u * (uint32_t)(c / CPH) + 16u * (uint32_t)(c % CPH);
  }
};

// barrier slots
enum : int {
  B_Q_FULL = 0, B_Q_EMPTY = 1, B_K_FULL = 2 /* x3 */, B_K_EMPTY = 5 /* x3 */,
  B_V_FULL = 8 /* x2 */, B_V_EMPTY = 10 /* x2 */, B_S_FULL = 12 /* x2: per row tile */,
  B_P_FULL = 14 /* x2 */, B_PV_DONE = 16 /* x2 */, B_O_EMPTY = 18 /* x2 */, B_DRAIN = 20,
  B_XCH = 21 /* x4: [row tile][parity], the split softmax's row exchange */,
  B_COUNT = 25
};

constexpr int kSoftWarps = 8 * kSplit;            // 4 * split per row tile
constexpr int kThreads = 32 * (2 + kSoftWarps);   // bf16 caches
constexpr int kThreadsF8 = kThreads + 128;        // E4M3 caches: + 4 converter warps

}  // namespace

struct PrefillParams {
  CUtensorMap tm_q;  // q as [T][Hq][D], box {64, G, 128/G}, 128B swizzle
  CUtensorMap tm_k;  // k_cache as [(blocks * Hkv * 16)][D], box {64, 16}
  CUtensorMap tm_v;
  const int32_t* qsl;
  const int32_t* seq_lens;
  const int32_t* block_tables;
  uint16_t* out;
  const WsHeader* header;
  const PrefillTile* tiles;
  int bt_stride, num_q_heads, num_kv_heads, num_blocks;
  float scale_log2;
  // cascade prefix pass
  int num_tokens, prefix_len, prefix_chunks, prefix_pairs, slot_floats;
  float* prefix_partials;
  // E4M3 caches (F8): raw codes and the output multiplier (1 for bf16)
  const unsigned char* k_cache8;
  const unsigned char* v_cache8;
  float v_scale;
  int overlap;  // PrefillLaunch::overlap
  unsigned long long* err;
};

// One work item as every role sees it.
struct Item {
  int req;    // block-table row (request 0 for the prefix pass)
  int kv;     // kv head
  int j0;     // first chunk token of the pair (prefill)
  int i0, n;  // key tiles i0 .. i0 + n - 1
  int L;      // keys that exist (sequence length; prefix length)
  int tok0;   // batch token of the pair's first row
  int chunk;  // key chunk (prefix pass)
};

template <int D, int G, bool PREFIX>
__device__ __forceinline__ Item get_item(const PrefillParams& p, int t) {
  using C = PCfg<D, G>;
  Item it;
  if constexpr (PREFIX) {
    const int nkt = (p.prefix_len + 127) / 128;
    const int per = (nkt + p.prefix_chunks - 1) / p.prefix_chunks;
    it.kv = t % p.num_kv_heads;
    const int rest = t / p.num_kv_heads;
    it.chunk = rest % p.prefix_chunks;
    it.req = 0;
    it.j0 = 0;
    it.i0 = it.chunk * per;
    it.n = min(per, nkt - it.i0);  // >= 1: the host picks chunks that are all non-empty
    it.L = p.prefix_len;
    it.tok0 = (rest / p.prefix_chunks) * 2 * C::TOK;
  } else {
    const PrefillTile tl = p.tiles[t];
    it.req = tl.req;
    it.kv = tl.kv;
    it.j0 = tl.j0;
    it.i0 = 0;
    it.n = tl.nkv;
    it.L = __ldg(p.seq_lens + tl.req);
    it.tok0 = __ldg(p.qsl + tl.req) + tl.j0;
    it.chunk = 0;
  }
  return it;
}

// One key row of an E4M3 tile widened to bf16 into a 128B-swizzled operand
// tile (row r: 16-byte unit u of 64-element chunk c lives at
// c * CHUNK + r * 128 + (u ^ (r & 7)) * 16). A row that is not a key of the
// sequence is written as zeros.
template <int D>
__device__ __forceinline__ void widen_e4m3_row(const unsigned char* src, bool valid,
                                               unsigned char* tile, int r) {
  constexpr int CHUNK = 128 * 128;
  uint4 raw[D / 16];
#pragma unroll
  for (int j = 0; j < D / 16; ++j)
    raw[j] = valid ? __ldg(reinterpret_cast<const uint4*>(src) + j) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
  for (int j = 0; j < D / 16; ++j) {
    const uint32_t w4[4] = {raw[j].x, raw[j].y, raw[j].z, raw[j].w};
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 a = e4m3x2_to_float2((uint16_t)(w4[i] & 0xffffu));
      const float2 b = e4m3x2_to_float2((uint16_t)(w4[i] >> 16));
      o[2 * i] = float2_to_bf16x2(a.x, a.y);
      o[2 * i + 1] = float2_to_bf16x2(b.x, b.y);
    }
    // elements 16j .. 16j+15: chunk 16j / 64, units (16j % 64) / 8 and the next
    const int c = (16 * j) / 64, u = ((16 * j) % 64) / 8;
    unsigned char* const rowp = tile + c * CHUNK + r * 128;
    *reinterpret_cast<uint4*>(rowp + ((u ^ (r & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
    *reinterpret_cast<uint4*>(rowp + (((u + 1) ^ (r & 7)) << 4)) =
        make_uint4(o[4], o[5], o[6], o[7]);
  }
}

// The r-th work item of CTA blockIdx.x among the g CTAs that take items.
// Items come sorted longest first; rounds of g items alternate direction (CTA b takes b, then 2g-1-b, then
// 2g+b, ...), so a CTA that drew a long item in one round draws a short one
// in the next instead of the next-longest.
__device__ __forceinline__ int snake_item(int r, int g) {
  const int b = (int)blockIdx.x;
  return r * g + ((r & 1) ? g - 1 - b : b);
}

template <int D, int G, bool PREFIX, bool F8>
__global__ void __launch_bounds__(F8 ? kThreadsF8 : kThreads, 1)
    pa_prefill_kernel(const __grid_constant__ PrefillParams p) {
  using C = PCfg<D, G>;
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;  // operand tiles need 1024-byte alignment
  unsigned char* const gbase = smem_raw + (base - raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t bar0 = base + C::OFF_BAR;
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(gbase + C::OFF_BAR + 8 * B_COUNT);

  if (threadIdx.x == 0) {
    for (int i = 0; i < B_COUNT; ++i) {
      // P_FULL and O_EMPTY are arrived at by the 128 threads of one warpgroup;
      // every other slot once, by an expect_tx arrive or an MMA commit.
      const bool by_threads = (i == B_P_FULL || i == B_P_FULL + 1 || i == B_O_EMPTY ||
                               i == B_O_EMPTY + 1 || (i >= B_XCH && i < B_XCH + 4));
      // E4M3 caches: the K / V stages are filled by the 4 converter warps
      const bool by_converters =
          F8 && ((i >= B_K_FULL && i < B_K_FULL + C::KSTAGES) ||
                 (i >= B_V_FULL && i < B_V_FULL + C::VSTAGES));
      mbar_init(bar0 + 8 * i, by_threads ? 128 * kSplit : (by_converters ? 4 : 1));
    }
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // The work list comes from the preceding (planner) grid. The prefix pass
  // needs none of it and waits only before it completes (see the end).
  if constexpr (!PREFIX) griddep_wait();
  int ntiles = PREFIX ? p.prefix_pairs * p.num_kv_heads * p.prefix_chunks : p.header->num_tiles;
  // CTAs taking items: all, or (overlapped mixed batch) the planner's share;
  // the others retire at once and leave their SMs to the split-KV grid,
  // which every CTA releases here rather than on completion
  int ctas = (int)gridDim.x;
  // Overlapped cascade: the prefix pass runs on a few SMs beside the suffix
  // split-KV grid, which needs the plan. One warp (the last softmax warp,
  // idle until the first scores) waits for the planner and then releases it.
  if (PREFIX && p.overlap && warp == 1 + kSoftWarps) {
    griddep_wait();
    griddep_launch_dependents();
  }
  if (!PREFIX && p.overlap) {
    const int c = __ldcg(&p.header->prefill_ctas);
    if (c > 0 && c < ctas) {
      ctas = c;
      griddep_launch_dependents();
    }
    if ((int)blockIdx.x >= ctas) ntiles = 0;
  }

  auto BAR = [&](int i) -> uint32_t { return bar0 + 8 * i; };
  auto wait = [&](int i, uint32_t parity) -> bool {
    if (mbar_wait_bounded(BAR(i), parity)) return true;
    report_error(p.err, PA_DEVERR_WAIT_TIMEOUT, 1000 + i);
    return false;
  };

  if (warp == 0) {
    // ======================= TMA producer =======================
    // Block ids are fetched 32 at a time (four key tiles), one group ahead;
    // lanes 0..7 each copy one 16-key block.
    int g = 0, it = 0;
    bool ok = true;
    for (int t = snake_item(it, ctas); ok && t < ntiles; t = snake_item(++it, ctas)) {
      const Item tl = get_item<D, G, PREFIX>(p, t);
      const int nb = (tl.L + kBlockSize - 1) / kBlockSize;
      const int32_t* const bt_row = p.block_tables + (size_t)tl.req * p.bt_stride;
      auto load_group = [&](int grp) -> int {  // blocks of key tiles i0 + 4 grp .. + 3
        const int b = tl.i0 * 8 + grp * 32 + lane;
        if (b >= nb) return -1;
        const int pid = __ldg(bt_row + b);
        if (pid < 0 || pid >= p.num_blocks) {
          report_error(p.err, PA_DEVERR_BLOCK_ID, b);
          return -1;
        }
        return pid;
      };
      int pid_cur = load_group(0);
      int pid_nxt = tl.n > 4 ? load_group(1) : -1;
      if (it > 0 && !wait(B_Q_EMPTY, (it - 1) & 1)) { ok = false; break; }
      if (lane == 0) {
        mbar_arrive_expect_tx(BAR(B_Q_FULL), 2 * C::Q_BYTES);
#pragma unroll
        for (int rt = 0; rt < 2; ++rt)
#pragma unroll
          for (int c = 0; c < C::NCH; ++c)
            tma_load_3d(base + C::OFF_Q + rt * C::Q_BYTES + c * C::CHUNK, &p.tm_q, c * 64,
                        tl.kv * G, tl.tok0 + rt * C::TOK, BAR(B_Q_FULL));
      }
      for (int i = 0; !F8 && i < tl.n; ++i, ++g) {  // E4M3: the converter warps load K/V
        if (i > 0 && (i & 3) == 0) {
          pid_cur = pid_nxt;
          pid_nxt = (i + 4 < tl.n) ? load_group((i >> 2) + 1) : -1;
        }
        const int ks = g % C::KSTAGES, vs = g % C::VSTAGES;
        const int pid = __shfl_sync(kAll, pid_cur, ((i & 3) << 3) + (lane & 7));
        const int nload = __popc(__ballot_sync(kAll, lane < 8 && pid >= 0));
        const int row = (pid * p.num_kv_heads + tl.kv) * kBlockSize;
        const bool mine = lane < 8 && pid >= 0;
        if (g >= C::KSTAGES && !wait(B_K_EMPTY + ks, ((g / C::KSTAGES) - 1) & 1)) { ok = false; break; }
        if (lane == 0) mbar_arrive_expect_tx(BAR(B_K_FULL + ks), nload * C::NCH * 2048);
        __syncwarp();
        if (mine) {
#pragma unroll
          for (int c = 0; c < C::NCH; ++c)
            tma_load_2d(base + C::OFF_K + ks * C::KV_BYTES + c * C::CHUNK + lane * 2048, &p.tm_k,
                        c * 64, row, BAR(B_K_FULL + ks));
        }
        if (g >= C::VSTAGES && !wait(B_V_EMPTY + vs, ((g / C::VSTAGES) - 1) & 1)) { ok = false; break; }
        if (lane == 0) mbar_arrive_expect_tx(BAR(B_V_FULL + vs), nload * C::NCH * 2048);
        __syncwarp();
        if (mine) {
#pragma unroll
          for (int c = 0; c < C::NCH; ++c)
            tma_load_2d(base + C::OFF_V + vs * C::KV_BYTES + c * C::CHUNK + lane * 2048, &p.tm_v,
                        c * 64, row, BAR(B_V_FULL + vs));
        }
      }
    }
  } else if (warp == 1) {
    // ======================= MMA issuer =======================
    constexpr uint32_t idesc_qk = idesc_bf16_f32(128, 128, false);
    constexpr uint32_t idesc_pv = idesc_bf16_f32(128, D, true);
    // Shared-memory descriptors differ only in their start address field
    // (address >> 4), so each MMA takes a base descriptor plus a constant.
    const uint64_t kmaj_base = smem_desc_sw128(base, 16, 1024);        // K-major (Q, K)
    const uint64_t vmaj_base = smem_desc_sw128(base, C::CHUNK, 1024);  // M/N-major (V)
    int gk = 0;   // key tiles whose S MMAs were issued
    int gv = 0;   // key tiles whose P*V MMAs were issued
    int np[2] = {0, 0};  // P_t events consumed
    int it = 0;
    bool ok = true;
    for (int t = snake_item(it, ctas); ok && t < ntiles; t = snake_item(++it, ctas)) {
      const Item tl = get_item<D, G, PREFIX>(p, t);
      const int L = tl.L;
      if (!wait(B_Q_FULL, it & 1)) { ok = false; break; }

      // S_rt(key tile of counter gk) for row tile rt
      auto issue_s = [&](int rt, bool last_of_item) -> bool {
        const int kst = gk % C::KSTAGES;
        if (rt == 0 && !wait(B_K_FULL + kst, (gk / C::KSTAGES) & 1)) return false;
        tc_fence_after();
        if (lane == 0) {
          const uint32_t d = tmem + C::TM_S + 128 * rt;
          const uint64_t a0 = kmaj_base + ((C::OFF_Q + rt * C::Q_BYTES) >> 4);
          const uint64_t b0 = kmaj_base + ((C::OFF_K + kst * C::KV_BYTES) >> 4);
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            const int off = ((ks / 4) * C::CHUNK + (ks % 4) * 32) >> 4;
            umma_bf16(d, a0 + off, b0 + off, idesc_qk, ks > 0 ? 1u : 0u);
          }
          umma_commit(BAR(B_S_FULL + rt));
          if (rt == 1) {
            umma_commit(BAR(B_K_EMPTY + kst));
            if (last_of_item) umma_commit(BAR(B_Q_EMPTY));
          }
        }
        __syncwarp();
        if (rt == 1) ++gk;
        return true;
      };
      // P_rt(key tile i) * V for row tile rt
      auto issue_pv = [&](int rt, int i) -> bool {
        const int vst = gv % C::VSTAGES;
        if (!wait(B_P_FULL + rt, np[rt] & 1)) return false;
        ++np[rt];
        if (rt == 0) {
          if (!wait(B_V_FULL + vst, (gv / C::VSTAGES) & 1)) return false;
          const int kv0 = (tl.i0 + i) * 128;
          if (!F8 && kv0 + 128 > L) {  // (the converters write such rows as zeros)
            // Rows of keys past the sequence end may hold anything (NaN too);
            // their P is 0, but 0 * NaN would poison O, so clear them.
            const int r0 = L - kv0;
            const int per_chunk = (128 - r0) * 8;  // 16-byte units
            for (int idx = lane; idx < per_chunk * C::NCH; idx += 32) {
              const int c = idx / per_chunk, rem = idx - c * per_chunk;
              const int row = r0 + (rem >> 3), u = rem & 7;
              *reinterpret_cast<uint4*>(gbase + C::OFF_V + vst * C::KV_BYTES + c * C::CHUNK +
                                        row * 128 + u * 16) = make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async_smem();
            __syncwarp();
          }
        }
        if (i == 0 && it > 0 && !wait(B_O_EMPTY + rt, (it - 1) & 1)) return false;
        tc_fence_after();
        if (lane == 0) {
          const uint32_t d = tmem + C::TM_O + 128 * rt;
          const uint32_t a_tm = tmem + C::TM_S + 128 * rt;  // P_rt: 64 columns of bf16 pairs
          const uint64_t b0 = vmaj_base + ((C::OFF_V + vst * C::KV_BYTES) >> 4);
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)  // keys 16 ks .. 16 ks + 15: 8 P columns
            umma_bf16_ta(d, a_tm + C::pcol(ks >> 1) + 8 * (ks & 1), b0 + ((ks * 2048) >> 4),
                         idesc_pv, (i > 0 || ks > 0) ? 1u : 0u);
          umma_commit(BAR(B_PV_DONE + rt));
          if (rt == 1) umma_commit(BAR(B_V_EMPTY + vst));
        }
        __syncwarp();
        if (rt == 1) ++gv;
        return true;
      };

      ok = issue_s(0, tl.n == 1) && issue_s(1, tl.n == 1);
      for (int i = 0; ok && i < tl.n; ++i) {
        const bool more = i + 1 < tl.n;
        const bool last_next = i + 2 == tl.n;
        ok = issue_pv(0, i);
        if (ok && more) ok = issue_s(0, last_next);
        if (ok) ok = issue_pv(1, i);
        if (ok && more) ok = issue_s(1, last_next);
      }
    }
    // every MMA issued above has completed before TMEM is released
    if (lane == 0) umma_commit(BAR(B_DRAIN));
    __syncwarp();
    mbar_wait_bounded(BAR(B_DRAIN), 0);
  } else if (warp < 2 + kSoftWarps) {
    // ======================= softmax + epilogue ==========================================
    // Row tile rt has warps 2 + 4*split*rt ...; within it, 4 warps per column
    // half hf (warp w reads TMEM lanes 32*(w%4) .. 32*(w%4)+31).
    const int sw = warp - 2;
    const int rt = sw / (4 * kSplit);     // row tile of this warp
    const int hf = (sw / 4) % kSplit;     // column half (0 without the split)
    const int q4 = warp & 3;              // TMEM lane quarter this warp may access
    const int m = q4 * 32 + lane;         // row == TMEM lane
    const uint32_t trow = ((uint32_t)(q4 * 32) << 16) + tmem;
    const uint32_t s_addr = trow + C::TM_S + 128 * rt;
    const uint32_t o_addr = trow + C::TM_O + 128 * rt;
    constexpr int OCH = D / 32 / kSplit;  // 32-column O chunks per thread
    float* const xch = reinterpret_cast<float*>(gbase + C::OFF_XCH);
    int nx = 0;  // exchanges done
    // Combine a per-thread row value with the other half's (max or sum). The
    // two halves meet on an mbarrier with a bounded wait (a half that gives up
    // cannot strand the other); exchange k uses barrier and buffer k % 2, so
    // a barrier is reused only after every thread has passed the other one.
    auto exchange = [&](float v, bool take_max, bool& good) -> float {
      if constexpr (kSplit == 1) {
        return v;
      } else {
        const int k = nx++;
        float* const xb = xch + ((rt * 2 + (k & 1)) * 2) * 128;
        xb[hf * 128 + m] = v;
        mbar_arrive(BAR(B_XCH + rt * 2 + (k & 1)));  // release: the store above is visible
        if (!wait(B_XCH + rt * 2 + (k & 1), (k >> 1) & 1)) {
          good = false;
          return v;
        }
        const float o = xb[(1 - hf) * 128 + m];
        return take_max ? fmaxf(v, o) : v + o;
      }
    };
    int ns = 0, it = 0;  // S_rt events consumed; work items done
    bool ok = true;
    for (int t = snake_item(it, ctas); ok && t < ntiles; t = snake_item(++it, ctas)) {
      const Item tl = get_item<D, G, PREFIX>(p, t);
      const int L = tl.L;
      int qlen = 0, j = 0, lim;
      if constexpr (PREFIX) {
        lim = L - 1;  // the whole prefix, for every row
      } else {
        qlen = __ldg(p.qsl + tl.req + 1) - __ldg(p.qsl + tl.req);
        const int ctx = L - qlen;
        j = tl.j0 + rt * C::TOK + m / G;  // chunk token of this row
        lim = min(ctx + j, L - 1);        // last key this row may see
      }
      float m_used = -INFINITY, l = 0.f;
      for (int i = 0; i < tl.n; ++i) {
        // S_rt(i) complete implies every earlier MMA is too: O_rt is stable
        // and P_rt(i-1) has been consumed.
        if (!wait(B_S_FULL + rt, ns & 1)) { ok = false; break; }
        ++ns;
        tc_fence_after();
        const int kv0 = (tl.i0 + i) * 128;
        const bool unmasked = __all_sync(kAll, kv0 + 127 <= lim);
        // pass 1: row max of the raw scores over visible keys
        float mx = -INFINITY;
#pragma unroll 1
        for (int cc = 0; cc < C::CPH; ++cc) {
          const int c = hf * C::CPH + cc;
          uint32_t r[32];
          tmem_ld32(s_addr + c * 32, r);
          tmem_wait_ld();
          if (unmasked) {
#pragma unroll
            for (int e = 0; e < 32; ++e) mx = fmaxf(mx, __uint_as_float(r[e]));
          } else {
            const int lim_c = lim - kv0 - c * 32;  // columns e <= lim_c are visible
#pragma unroll
            for (int e = 0; e < 32; ++e) mx = fmaxf(mx, e <= lim_c ? __uint_as_float(r[e]) : -INFINITY);
          }
        }
        mx = exchange(mx, true, ok);         // the whole row's max
        if (!ok) break;
        const float mt = mx * p.scale_log2;  // -inf stays -inf
        float alpha = 1.f;
        bool resc = false;
        if (i == 0) {
          m_used = mt;  // the item's first key is always visible: finite
        } else if (mt > m_used + 8.f) {
          alpha = exp2f(m_used - mt);
          m_used = mt;
          resc = true;
        }
        if (__any_sync(kAll, resc)) {
#pragma unroll 1
          for (int oc = 0; oc < OCH; ++oc) {
            const int c = hf * OCH + oc;
            uint32_t o[32];
            tmem_ld32(o_addr + c * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32(o_addr + c * 32, o);
          }
          tmem_wait_st();
        }
        l *= alpha;
        // pass 2: P = exp2(s * scale - m) as bf16 pairs, written over this
        // thread's own S columns: chunk c's 16 P columns start at pcol(c),
        // which only covers S columns this thread has already read.
        const float nm = -m_used;
        const float sc = p.scale_log2;
        float l2[2] = {0.f, 0.f};  // two partial sums: shorter dependency chains
#pragma unroll 1
        for (int cc = 0; cc < C::CPH; ++cc) {
          const int c = hf * C::CPH + cc;
          uint32_t r[32];
          tmem_ld32(s_addr + c * 32, r);
          tmem_wait_ld();
          uint32_t w[16];
          if (unmasked) {
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const float p0 = ex2_approx(fmaf(__uint_as_float(r[2 * e]), sc, nm));
              const float p1 = ex2_approx(fmaf(__uint_as_float(r[2 * e + 1]), sc, nm));
              l2[e & 1] += p0 + p1;
              w[e] = float2_to_bf16x2(p0, p1);
            }
          } else {
            const int lim_c = lim - kv0 - c * 32;
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const float p0 = 2 * e <= lim_c ? ex2_approx(fmaf(__uint_as_float(r[2 * e]), sc, nm)) : 0.f;
              const float p1 =
                  2 * e + 1 <= lim_c ? ex2_approx(fmaf(__uint_as_float(r[2 * e + 1]), sc, nm)) : 0.f;
              l2[e & 1] += p0 + p1;
              w[e] = float2_to_bf16x2(p0, p1);
            }
          }
          tmem_st16(s_addr + C::pcol(c), w);
        }
        l += l2[0] + l2[1];
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(BAR(B_P_FULL + rt));
      }
      if (!ok) break;
      // ---- epilogue: O / l -> bf16 rows of out ----
      if (!wait(B_PV_DONE + rt, (ns - 1) & 1)) { ok = false; break; }
      tc_fence_after();
      l = exchange(l, false, ok);  // the whole row's sum
      if (!ok) break;
      if constexpr (PREFIX) {
        // fp32 partial of (chunk, token, kv head), head m % G of the slot
        const int tok = tl.tok0 + rt * C::TOK + m / G;
        const int h = m % G;
        const bool store = tok < p.num_tokens;
        float* const slot = p.prefix_partials +
                            (((size_t)tl.chunk * p.num_tokens + (store ? tok : 0)) *
                                 p.num_kv_heads + tl.kv) * p.slot_floats;
        if (store && hf == 0) {
          __stcg(slot + h, m_used);
          __stcg(slot + G + h, l);
        }
#pragma unroll 1
        for (int oc = 0; oc < OCH; ++oc) {
          const int c = hf * OCH + oc;
          uint32_t o[32];
          tmem_ld32(o_addr + c * 32, o);
          tmem_wait_ld();
          if (store) {
            float* const dst = slot + 16 + h * D + c * 32;
#pragma unroll
            for (int v = 0; v < 8; ++v)
              __stcg(reinterpret_cast<float4*>(dst + 4 * v),
                     make_float4(__uint_as_float(o[4 * v]), __uint_as_float(o[4 * v + 1]),
                                 __uint_as_float(o[4 * v + 2]), __uint_as_float(o[4 * v + 3])));
          }
        }
        tc_fence_before();
        mbar_arrive(BAR(B_O_EMPTY + rt));
        continue;
      }
      const float inv = p.v_scale / l;
      const bool store = j < qlen;
      uint16_t* const orow =
          p.out + ((size_t)(tl.tok0 - tl.j0 + j) * p.num_q_heads + (size_t)tl.kv * G + (m % G)) * D;
#pragma unroll 1
      for (int oc = 0; oc < OCH; ++oc) {
        const int c = hf * OCH + oc;
        uint32_t o[32];
        tmem_ld32(o_addr + c * 32, o);
        tmem_wait_ld();
        if (store) {
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint4 pk;
            pk.x = float2_to_bf16x2(__uint_as_float(o[8 * v + 0]) * inv, __uint_as_float(o[8 * v + 1]) * inv);
            pk.y = float2_to_bf16x2(__uint_as_float(o[8 * v + 2]) * inv, __uint_as_float(o[8 * v + 3]) * inv);
            pk.z = float2_to_bf16x2(__uint_as_float(o[8 * v + 4]) * inv, __uint_as_float(o[8 * v + 5]) * inv);
            pk.w = float2_to_bf16x2(__uint_as_float(o[8 * v + 6]) * inv, __uint_as_float(o[8 * v + 7]) * inv);
            *reinterpret_cast<uint4*>(orow + c * 32 + 8 * v) = pk;
          }
        }
      }
      tc_fence_before();
      mbar_arrive(BAR(B_O_EMPTY + rt));
    }
  } else if constexpr (F8) {
    // ======================= E4M3 converters (warps 10-13) =======================
    const int r = threadIdx.x - kThreads;  // key row of the tile, 0..127 (converter warps)
    int g = 0, it = 0;
    bool ok = true;
    for (int t = snake_item(it, ctas); ok && t < ntiles; t = snake_item(++it, ctas)) {
      const Item tl = get_item<D, G, PREFIX>(p, t);
      const int32_t* const bt_row = p.block_tables + (size_t)tl.req * p.bt_stride;
      for (int i = 0; i < tl.n; ++i, ++g) {
        const int key = (tl.i0 + i) * 128 + r;
        bool valid = key < tl.L;
        size_t src = 0;
        if (valid) {
          const int pid = __ldg(bt_row + key / kBlockSize);
          if (pid < 0 || pid >= p.num_blocks) {
            report_error(p.err, PA_DEVERR_BLOCK_ID, key / kBlockSize);
            valid = false;
          } else {
            src = (((size_t)pid * p.num_kv_heads + tl.kv) * kBlockSize + (key % kBlockSize)) * D;
          }
        }
        const int ks = g % C::KSTAGES, vs = g % C::VSTAGES;
        if (g >= C::KSTAGES && !wait(B_K_EMPTY + ks, ((g / C::KSTAGES) - 1) & 1)) { ok = false; break; }
        widen_e4m3_row<D>(p.k_cache8 + src, valid, gbase + C::OFF_K + ks * C::KV_BYTES, r);
        fence_proxy_async_smem();  // generic-proxy stores -> visible to the tensor core
        __syncwarp();
        if (lane == 0) mbar_arrive(BAR(B_K_FULL + ks));
        if (g >= C::VSTAGES && !wait(B_V_EMPTY + vs, ((g / C::VSTAGES) - 1) & 1)) { ok = false; break; }
        widen_e4m3_row<D>(p.v_cache8 + src, valid, gbase + C::OFF_V + vs * C::KV_BYTES, r);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(BAR(B_V_FULL + vs));
      }
    }
  }

  if constexpr (PREFIX) {
    // The split-KV grid launched after this one may start now; this grid does
    // not complete before the planner (and the KV write before it) has, so a
    // dependent that waits for this grid sees the plan too. (The prefill-chunk
    // grid releases its dependent only by completing: triggering here too
    // measured 0.53 vs 0.435 ms per mixed step.) Overlapped, it did both at
    // the top.
    if (!p.overlap) {
      griddep_launch_dependents();
      griddep_wait();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------------------
namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool get_encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode != nullptr;
}

bool encode_bf16(CUtensorMap* m, int rank, const void* ptr, const cuuint64_t* dims,
                 const cuuint64_t* strides_bytes, const cuuint32_t* box,
                 CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  const CUresult r = g_encode(m, dtype, rank, const_cast<void*>(ptr),
                              dims, strides_bytes, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace

bool encode_tmap_bf16_2d(void* tmap, const void* ptr, uint64_t inner, uint64_t rows,
                         uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_rows) {
  if (!get_encoder()) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
  const cuuint64_t str[1] = {(cuuint64_t)row_stride_bytes};
  const cuuint32_t box[2] = {box_inner, box_rows};
  return encode_bf16(static_cast<CUtensorMap*>(tmap), 2, ptr, dims, str, box);
}

namespace {
bool encode_tmap_any(void* tmap, int rank, const void* ptr, const uint64_t* dims,
                     const uint64_t* strides_bytes, const uint32_t* box, CUtensorMapDataType dt) {
  if (!get_encoder() || rank < 1 || rank > 5) return false;
  cuuint64_t d[5], st[4];
  cuuint32_t b[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = (cuuint64_t)dims[i];
    b[i] = (cuuint32_t)box[i];
    if (i + 1 < rank) st[i] = (cuuint64_t)strides_bytes[i];
  }
  return encode_bf16(static_cast<CUtensorMap*>(tmap), rank, ptr, d, st, b, dt);
}
}  // namespace

bool encode_tmap_bf16(void* tmap, int rank, const void* ptr, const uint64_t* dims,
                      const uint64_t* strides_bytes, const uint32_t* box) {
  return encode_tmap_any(tmap, rank, ptr, dims, strides_bytes, box,
                         CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);
}

bool encode_tmap_u8(void* tmap, int rank, const void* ptr, const uint64_t* dims,
                    const uint64_t* strides_bytes, const uint32_t* box) {
  return encode_tmap_any(tmap, rank, ptr, dims, strides_bytes, box, CU_TENSOR_MAP_DATA_TYPE_UINT8);
}

namespace {

template <int D, int G, bool PREFIX, bool F8>
cudaError_t launch_prefill_t(const PrefillLaunch& a, int num_sms, cudaStream_t s) {
  using C = PCfg<D, G>;
  PrefillParams p;
  {
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)a.num_q_heads, (cuuint64_t)a.num_tokens};
    const cuuint64_t str[2] = {(cuuint64_t)D * 2, (cuuint64_t)a.num_q_heads * D * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)G, (cuuint32_t)C::TOK};
    if (!encode_bf16(&p.tm_q, 3, a.q, dims, str, box)) return cudaErrorInvalidValue;
  }
  if (!F8) {  // E4M3 K/V are loaded by the converter warps, not by TMA
    const cuuint64_t rows = (cuuint64_t)a.num_blocks * a.num_kv_heads * kBlockSize;
    const cuuint64_t dims[2] = {(cuuint64_t)D, rows};
    const cuuint64_t str[1] = {(cuuint64_t)D * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)kBlockSize};
    if (!encode_bf16(&p.tm_k, 2, a.k_cache, dims, str, box)) return cudaErrorInvalidValue;
    if (!encode_bf16(&p.tm_v, 2, a.v_cache, dims, str, box)) return cudaErrorInvalidValue;
  }
  p.qsl = a.qsl;
  p.seq_lens = a.seq_lens;
  p.block_tables = a.block_tables;
  p.out = a.out;
  p.header = a.header;
  p.tiles = a.tiles;
  p.bt_stride = a.bt_stride;
  p.num_q_heads = a.num_q_heads;
  p.num_kv_heads = a.num_kv_heads;
  p.num_blocks = a.num_blocks;
  p.scale_log2 = a.scale_log2;
  p.err = a.err;
  p.num_tokens = a.num_tokens;
  p.prefix_len = a.prefix_len;
  p.prefix_chunks = a.prefix_chunks;
  p.prefix_pairs = prefix_pairs(a.num_tokens, G);
  p.slot_floats = a.slot_floats;
  p.prefix_partials = a.prefix_partials;
  p.k_cache8 = F8 ? static_cast<const unsigned char*>(a.k_cache) : nullptr;
  p.v_cache8 = F8 ? static_cast<const unsigned char*>(a.v_cache) : nullptr;
  p.v_scale = F8 ? a.v_scale : 1.f;
  p.overlap = a.overlap;
  int grid = num_sms;
  if (PREFIX) {
    const int items = p.prefix_pairs * a.num_kv_heads * a.prefix_chunks;
    grid = items < num_sms ? items : num_sms;
    // overlapped cascade: the pass keeps to its share of the SMs
    if (a.overlap && a.prefix_ctas > 0 && a.prefix_ctas < grid) grid = a.prefix_ctas;
  }

  auto kern = pa_prefill_kernel<D, G, PREFIX, F8>;
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(F8 ? kThreadsF8 : kThreads);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace

template <bool PREFIX, bool F8>
cudaError_t launch_prefill_mode(const PrefillLaunch& a, int num_sms, cudaStream_t s) {
  const int G = a.num_q_heads / a.num_kv_heads;
  if (a.head_dim == 128) {
    switch (G) {
      case 1: return launch_prefill_t<128, 1, PREFIX, F8>(a, num_sms, s);
      case 2: return launch_prefill_t<128, 2, PREFIX, F8>(a, num_sms, s);
      case 4: return launch_prefill_t<128, 4, PREFIX, F8>(a, num_sms, s);
      case 8: return launch_prefill_t<128, 8, PREFIX, F8>(a, num_sms, s);
    }
  } else if (a.head_dim == 64) {
    switch (G) {
      case 1: return launch_prefill_t<64, 1, PREFIX, F8>(a, num_sms, s);
      case 2: return launch_prefill_t<64, 2, PREFIX, F8>(a, num_sms, s);
      case 4: return launch_prefill_t<64, 4, PREFIX, F8>(a, num_sms, s);
      case 8: return launch_prefill_t<64, 8, PREFIX, F8>(a, num_sms, s);
    }
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_prefill(const PrefillLaunch& a, int num_sms, cudaStream_t s) {
  if (!get_encoder()) return cudaErrorNotSupported;
  if (a.kv_fp8) {
    if (a.prefix_len > 0) return cudaErrorNotSupported;  // no FP8 cascade
    return launch_prefill_mode<false, true>(a, num_sms, s);
  }
  return a.prefix_len > 0 ? launch_prefill_mode<true, false>(a, num_sms, s)
                          : launch_prefill_mode<false, false>(a, num_sms, s);
}

}  // namespace pa
