// Chunked KDA on the 5th-generation tensor cores (tcgen05 MMAs with TMEM accumulators,
// TMA-fed shared memory) for bf16 q/k/v with dk = dv = 128, as two kernels.
//
// Chunk algebra. For a chunk of C = 64 tokens entering with state S (rows = key channels),
// gamma = cumsum(g) over the chunk (per channel, natural log), the gated delta rule unrolls to
//   U   = U0 - W S                               (the chunk's corrected values)
//   O   = Q'' S + O0                             (the chunk's outputs, scale folded in)
//   S_C = Diag(e^gamma_C) S + Kb'^T U            (the state after the chunk)
// with every other factor independent of S:
//   T   = (I + strict_lower(Diag(beta) Kh Kb^T))^-1,   TB = T Diag(beta)
//   K'  = k e^gamma,  Kb' = k e^(gamma_C - gamma),  W = TB K',  U0 = TB V
//   Aqk = tril(Qh Kb^T)  (query-key products weighted by e^(gamma_t - gamma_i), i <= t)
//   P   = Aqk TB,  Q'' = scale (q e^gamma - P K'),  O0 = scale P V
// where Kh = k e^(gamma - rho), Qh = q e^(gamma - rho), Kb = k e^(rho - gamma) and, per
// channel, rho = gamma_C / 2: in this midpoint frame every factor stays within e^(+-80) as long
// as the channel decays by at most 160 nats over the chunk. A channel that decays more (a
// "strong" channel) takes frame rho = 0 and no share in the Kh Kb^T product (its Kb is zero);
// its share of A_kk and A_qk is added exactly on CUDA cores from pairwise factors
// e^(gamma_t - gamma_i) <= 1, and its Kb' is formed directly. Every g <= 0 is thus exact up
// to rounding; chunks without strong channels never enter that code.
//
// Kernel 1 (prep) computes the state-independent factors of every (chunk, head) in parallel
// (persistent CTAs, one item at a time, the next item's loads in flight) and writes them to a
// workspace record. Kernel 2 (state) walks each range's chunks in order for one (range, head,
// 128-column tile of the state) with the transposed state S^T in two TMEM buffers: per chunk
// one N = 128 product X^T = S^T [W; Q'']^T, the U update and the outputs on CUDA cores, the
// decayed state S^T Diag(e^gamma_C) written into the other buffer next to X, and one N = 128
// product U^T Kb' accumulated onto it, with the records streamed in by TMA two chunks ahead.
// In package mode kernel 2 runs the same chunks on the M or the D half of the
// augmented state [M | D] (identity / zero start; M columns see zero values) and writes no
// outputs. A fused cooperative launch runs both kernels' work side by side for few walks.
//
// MMAs are kind::tf32 with fp32 accumulation, except U0^T = V^T TB^T, a kind::f16 product of
// the bf16 v staging (read MN-major) and TB split into bf16 hi and lo parts. Every other
// shared-memory operand is K-major in the 128-byte swizzle; operands needed in the other
// orientation are written transposed by the threads that produce them or staged in TMEM.
// Waits on mbarriers are bounded (2 s of globaltimer); on expiry a CTA raises
// KDA_STATUS_TIMEOUT, drains its own MMAs and copies (bounded), frees its TMEM and returns.
#include <cuda.h>

#include <algorithm>

#include "kda_internal.cuh"
#include "ptx.cuh"

namespace kda {
namespace {

using namespace ptx;

constexpr int C = kChunk;  // 64 tokens per chunk
constexpr int DK = 128;
constexpr int kThreads = 256;
constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------- workspace record
// Per item (chunk slot, head):
//   wq  [128][128] fp32  rows 0..63 W, rows 64..127 Q''   (row = token, column = channel)
//   kbt [128][64]  fp32  Kb'^T                            (row = channel, column = token)
//   u0  [16][128][4] fp32 U0^T, tokens 4b .. 4b+3 of value column n at [b][n]
//   o0  [8][128][8]  bf16 O0^T, tokens 8b .. 8b+7 of value column n at [b][n]
// (U0^T and O0^T are interleaved so that 32 consecutive value columns read one token group as
// one contiguous 512-byte run.)
//   dec [128]      fp32  e^gamma_C
// Chunk j of range i (starting at token b_i) has slot floor(b_i / C) + i + j: distinct for
// distinct chunks of valid ordered ranges, and below floor(T / C) + n_ranges.
constexpr size_t kWqBytes = 128 * 128 * 4;
constexpr size_t kKbtBytes = 128 * 64 * 4;
constexpr size_t kU0Bytes = 128 * 64 * 4;
constexpr size_t kO0Bytes = 128 * 64 * 2;
constexpr size_t kDecBytes = 128 * 4;
constexpr size_t kItemBytes = kWqBytes + kKbtBytes + kU0Bytes + kO0Bytes + kDecBytes;

struct Ws {
  float* wq;
  float* kbt;
  float* u0;
  __nv_bfloat16* o0;
  float* dec;
};

__device__ __forceinline__ void cta_sync() {
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
}

__device__ __forceinline__ float* f32at(uint8_t* base, uint32_t off) {
  return reinterpret_cast<float*>(base + off);
}

// 8 consecutive bf16 (one 16-byte chunk) -> fp32
__device__ __forceinline__ void unpack8(const uint4 r, float* x) {
  const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// Chunk of an item; false for a slot that holds no chunk (or an invalid range).
__device__ bool item_chunk(const ChunkParams& p, int item, int& t0, int& n, int& h) {
  const int slot = item / p.H;
  h = item - slot * p.H;
  int i = 0;
  if (p.offsets) {  // largest i with floor(b_i / C) + i <= slot
    int lo = 0, hi = p.n_ranges - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (p.offsets[mid] / C + mid <= slot) lo = mid;
      else hi = mid - 1;
    }
    i = lo;
  }
  const int b = p.offsets ? p.offsets[i] : 0;
  const int e = p.offsets ? p.offsets[i + 1] : p.total_tokens;
  if (b < 0 || e > p.total_tokens || e < b) return false;
  const int j = slot - (b / C + i);
  if (j < 0) return false;
  t0 = b + j * C;
  if (t0 >= e) return false;
  n = min(C, e - t0);
  return true;
}

// ============================================================================ kernel 1: prep
// shared memory (byte offsets from a 1024-byte aligned base)
constexpr uint32_t P_STG_Q = 0;         // 2 x [64 tok][64 ch] bf16, 128-byte swizzle
constexpr uint32_t P_STG_K = 16384;
constexpr uint32_t P_STG_V = 32768;
constexpr uint32_t P_STG_G = 49152;     // 4 x [64 tok][32 ch] fp32, 128-byte swizzle
constexpr uint32_t P_STG_B = 81920;     // [64 tok][4 heads] fp32
constexpr uint32_t P_KB = 82944;        // Kb [64 tok][128 ch] fp32 (4 K-blocks of 8 KiB)
constexpr uint32_t P_KB_KB = 8192;
constexpr uint32_t P_BE = P_KB + 32768;  // K'^T [128][64 tok] fp32 (2 K-blocks)
constexpr uint32_t P_BE_KB = 16384;
constexpr uint32_t P_TBT = P_BE + 32768;  // TB^T [64][64] fp32 (2 K-blocks of 8 KiB)
constexpr uint32_t P_TBT_KB = 8192;
// After the solve, the Kb buffer holds TB as bf16 hi and lo parts ([t][t'] rows of 128 B,
// K-major over t'; TB = hi + lo to 2^-17) and tril(A_qk) row-major fp32: the B operands of
// U0^T = V^T TB^T (a kind::f16 product whose A operand is the bf16 V staging itself, read
// MN-major) and of O0^T = U0^T A_qk^T.
constexpr uint32_t P_TBN = P_KB;
constexpr uint32_t P_PN = P_KB + 16384;
constexpr uint32_t P_XTRA = P_TBT + 16384;
constexpr int LA = 68;                    // padded row length of the solve scratch
constexpr uint32_t SCR_A = P_KB;          // beta_r A_kk [64][68] (Kb is dead by then)
constexpr uint32_t SCR_X = P_XTRA;        // (I + A_kk)^-1 [64][68]
constexpr uint32_t SCR_P = P_XTRA + 64 * LA * 4;  // 8 warps x [16][8]
constexpr uint32_t P_MISC = SCR_P + 8 * 128 * 4;
// Workspace-record staging for the bulk-tensor stores (U0^T and O0^T go straight from
// registers to their interleaved records): W and Q'' as 4 boxes of [64 rows][32] fp32 in the
// 128-byte swizzle. Q'' over K'^T and W over TB^T and the solve's X scratch, all dead once R
// is complete (the O0^T product may still be reading tril(A_qk) in the Kb buffer). Only Q''
// (stored first) has to have left before the next item's operands are written; W's region is
// next written by that item's solve.
constexpr uint32_t ST_Q = P_BE;
constexpr uint32_t ST_W = P_TBT;
static_assert(ST_Q + 32768 <= P_TBT && ST_W + 32768 <= SCR_P, "record staging overflow");
constexpr uint32_t P_SMEM = P_MISC + 2048 + 1024;
static_assert(64 * LA * 4 <= 32768, "A_kk scratch must fit in the Kb buffer");
static_assert(P_KB % 1024 == 0 && P_BE % 1024 == 0 && P_TBT % 1024 == 0, "alignment");

// TMEM columns (512)
constexpr uint32_t TM_XA = 0;    // 128: [Kh ; Qh] (lanes = tokens), the A operand of A1
constexpr uint32_t TM_A1 = 128;  // 64: [Kh ; Qh] Kb^T -> [0 ; Aqk], the A operand of P
constexpr uint32_t TM_E = 192;   // 64: [TB ; 0] + [0 ; Aqk] TB = [TB ; P], the A operand of E
constexpr uint32_t TM_R = 256;   // 128: [0 ; -Q'] + [TB ; P] K' = [W ; P K' - Q']
constexpr uint32_t TM_U0T = 384;  // 64: V^T TB^T = U0^T (lanes = value columns)
constexpr uint32_t TM_O0T = 448;  // 64: U0^T A_qk^T = (A_qk TB V)^T = (P V)^T

struct PrepMisc {
  uint64_t bar_tma, bar_v, bar_a, bar_p, bar_u, bar_r, bar_e, bar_drain;
  uint32_t tmem_base;
  int abort;
  int nxt[4];  // item, t0, n, head of the item whose loads are in flight
  // fused launch: items whose records are complete, handed from the loader thread to the
  // publishing warp (ring of 4; pub_head counts the items handed over, pub_tail the flags
  // published; item -1 ends the stream)
  int pub_ring[4];
  uint32_t pub_head, pub_tail;
  // the item's strong channels (bit c % 32 of word c / 32): those whose decay over the chunk
  // exceeds kMaxChunkDecay nats, which the midpoint frame cannot hold
  uint32_t smask[4];
  // read with 16-byte vector loads
  alignas(16) float part[2][DK];
  alignas(16) float erho[DK];
  alignas(16) float beta[C];
};
static_assert(sizeof(PrepMisc) <= 2048, "misc overflow");
static_assert(offsetof(PrepMisc, part) % 16 == 0 && offsetof(PrepMisc, erho) % 16 == 0 &&
                  offsetof(PrepMisc, beta) % 16 == 0,
              "vector-loaded arrays must be 16-byte aligned");

// The prep CTA's 256 threads synchronise on named barrier 1 (a fused launch runs them next to
// its publishing warp and three idle warps).
__device__ __forceinline__ void pbar() { asm volatile("bar.sync 1, 256;" ::: "memory"); }
__device__ __forceinline__ void psync() {
  tc_fence_before();
  pbar();
  tc_fence_after();
}

// Processes items first, first + stride, ... (those holding a chunk). With `flags`, sets
// flags[item] (release, gpu scope) once the item's record is complete in global memory.
__device__ __forceinline__ void prep_run(const ChunkParams& p, const CUtensorMap& tmq,
                                         const CUtensorMap& tmk, const CUtensorMap& tmv,
                                         const CUtensorMap& tmg, const CUtensorMap& tmb,
                                         const CUtensorMap& twq_st, const Ws& ws,
                                         const int n_items, const int first, const int stride,
                                         uint32_t* flags) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  PrepMisc* misc = reinterpret_cast<PrepMisc*>(sm + P_MISC);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int qd = warp & 3;    // TMEM lane quarter
  const int chh = warp >> 2;  // half of the columns / channels
  const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
  const bool need_out = p.package == 0;
  const uint32_t tx_bytes = (need_out ? 16384u : 0u) + 16384u + 32768u + 1024u;  // q, k, g, beta

  if (warp == 0) {
    tmem_alloc(&misc->tmem_base, 512);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(&misc->bar_tma, 1);
    mbar_init(&misc->bar_v, 1);
    mbar_init(&misc->bar_a, 1);
    mbar_init(&misc->bar_p, 1);
    mbar_init(&misc->bar_u, 1);
    mbar_init(&misc->bar_r, 1);
    mbar_init(&misc->bar_e, 1);
    mbar_init(&misc->bar_drain, 2);  // both MMA-issuing threads drain into it
    misc->abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmk);
    tma_prefetch_desc(&tmv);
    tma_prefetch_desc(&tmg);
    tma_prefetch_desc(&tmb);
    if (need_out) tma_prefetch_desc(&tmq);
  }
  psync();
  const uint32_t tbase = misc->tmem_base;
  const uint32_t sbase = smem_u32(sm);

  auto issue_tma = [&](int t0, int hh) {
    mbar_arrive_expect_tx(&misc->bar_tma, tx_bytes);
    if (need_out) {
      tma_load_3d(sm + P_STG_Q, &tmq, &misc->bar_tma, 0, hh, t0);
      tma_load_3d(sm + P_STG_Q + 8192, &tmq, &misc->bar_tma, 64, hh, t0);
    }
    tma_load_3d(sm + P_STG_K, &tmk, &misc->bar_tma, 0, hh, t0);
    tma_load_3d(sm + P_STG_K + 8192, &tmk, &misc->bar_tma, 64, hh, t0);
#pragma unroll
    for (int kb = 0; kb < 4; ++kb)
      tma_load_3d(sm + P_STG_G + kb * 8192, &tmg, &misc->bar_tma, kb * 32, hh, t0);
    tma_load_2d(sm + P_STG_B, &tmb, &misc->bar_tma, hh & ~3, t0);
  };
  // v has its own barrier: its staging is the A operand of the U0^T product, so the next
  // item's v is loaded once that product is complete
  auto issue_v = [&](int t0, int hh) {
    mbar_arrive_expect_tx(&misc->bar_v, 16384u);
    tma_load_3d(sm + P_STG_V, &tmv, &misc->bar_v, 0, hh, t0);
    tma_load_3d(sm + P_STG_V + 8192, &tmv, &misc->bar_v, 64, hh, t0);
  };
  // thread 0: finds this CTA's next item holding a chunk, from `from` on, and issues its loads
  auto advance = [&](int from) {
    int it = from, t0 = 0, n = 0, hh = 0;
    while (it < n_items && !item_chunk(p, it, t0, n, hh)) it += stride;
    misc->nxt[0] = it;
    misc->nxt[1] = t0;
    misc->nxt[2] = n;
    misc->nxt[3] = hh;
    if (it < n_items) issue_tma(t0, hh);
    return it < n_items;
  };
  // Loads are issued by the loader thread, MMAs by thread 0, so that the next item's loads go
  // out while thread 0 is issuing the A1 product. The loader sits in warp 5, the warp with the
  // least work on the item's critical path (its key rows do the light operand iterations first,
  // and it has no share in the solve's substitution or the extraction's longest rows).
  constexpr int kLoader = 160;
  bool tma_out = false;  // loader: a load is in flight, completing phase parity tma_par
  uint32_t tma_par = 0;
  bool v_issued = false;  // loader: a v load was issued, the last completing phase v_par
  uint32_t v_par = 0;
  int prev_item = -1;    // loader: item whose record's store group is the latest but one
  uint32_t pub_n = 0;    // loader: items handed to the publishing warp
  // loader: hands an item (or -1, the end) to the publishing warp of a fused launch
  auto hand_over = [&](int it) {
    const uint64_t t0 = globaltimer_ns();
    while (pub_n - ld_acquire_cta(&misc->pub_tail) >= 4u) {  // ring full: bounded wait
      if (globaltimer_ns() - t0 > 1000000000ull) { misc->abort = 1; return; }
      __nanosleep(32);
    }
    misc->pub_ring[pub_n & 3] = it;
    st_release_cta(&misc->pub_head, ++pub_n);
  };
  if (tid == kLoader) {
    tma_out = advance(first);
    if (tma_out) {
      issue_v(misc->nxt[1], misc->nxt[3]);
      v_issued = true;
    }
  }
  psync();

  uint32_t k_it = 0;
  for (;;) {
    const int item = misc->nxt[0];
    if (item >= n_items) break;
    const int n = misc->nxt[2], h = misc->nxt[3];
    const uint32_t par = k_it & 1u;
    // ================= decay prefix (channel role: channel c, token half)
    if (!mbar_wait(&misc->bar_tma, par)) misc->abort = 1;
    else if (tid == kLoader) tma_out = false;
    {
      const int c = tid & (DK - 1), half = tid >> 7;
      const uint32_t gbase =
          P_STG_G + (uint32_t)(c >> 5) * 8192u + (uint32_t)(c & 3) * 4u + half * 4096u;
      const uint32_t xg = (uint32_t)(c & 31) >> 2;
      float gl[32];
      float acc = 0.0f;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const uint32_t off = gbase + (uint32_t)i * 128u + ((xg ^ (uint32_t)(i & 7)) << 4);
        gl[i] = (half * 32 + i < n) ? *f32at(sm, off) * kLog2e : 0.0f;
        acc += gl[i];
      }
      misc->part[half][c] = acc;
      if (tid < C) misc->beta[tid] = (tid < n) ? f32at(sm, P_STG_B)[tid * 4 + (h & 3)] : 0.0f;
      pbar();
      const float p0 = misc->part[0][c], p1 = misc->part[1][c];
      const float gsum = p0 + p1;  // gamma_C, log2 units
      // A strong channel (decay over the chunk beyond kMaxChunkDecay nats) takes frame 0: it
      // is left out of the A1 product and its share of A_kk / A_qk is computed exactly below.
      const bool strong = !(gsum >= -kMaxChunkDecay * kLog2e);
      const float rho2 = strong ? 0.0f : 0.5f * gsum;  // log2 units
      if (half == 0) {
        misc->erho[c] = ex2_approx(rho2);
        ws.dec[(size_t)item * DK + c] = ex2_approx(gsum);
        const uint32_t m = __ballot_sync(0xffffffffu, strong);  // warps 0..3: channels 32 w ..
        if (lane == 0) misc->smask[warp] = m;
      }
      // gamma - rho (log2 units) in place of g: each element has one owner
      float gam = half ? p0 : 0.0f;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        gam += gl[i];
        *f32at(sm, gbase + (uint32_t)i * 128u + ((xg ^ (uint32_t)(i & 7)) << 4)) = gam - rho2;
      }
    }
    if (tid == kLoader) bulk_wait_read1();  // the previous record's Q'' has left its staging
    pbar();
    const uint32_t* smask = misc->smask;
    const bool any_strong = (smask[0] | smask[1] | smask[2] | smask[3]) != 0u;
    // ================= operands (row role: token t; key rows in warps 0,1,4,5, query rows
    // in warps 2,3,6,7; channel half chh)
    // Of the 64 channels of its half, the thread forms Kb, Kb'^T and K'^T for 32 (offset hoff):
    // key rows the first 32 in half 0 and the last 32 in half 1, query rows the others. Warps
    // w and w + 4 share an SMSP, so each SMSP runs one warp's heavy iterations next to the
    // other's light ones.
    const int hoff = ((qd < 2) == (chh == 0)) ? 0 : 32;
    {
      const int t = (qd & 1) * 32 + lane;
      const bool valid = t < n;
      const uint32_t tsw = (uint32_t)(t & 7);
      const uint32_t grow = P_STG_G + (uint32_t)t * 128u;
      const uint32_t brow = (uint32_t)t * 128u;
      // Kb (the B operand of A1), Kb'^T (workspace) and K'^T (B operand of R) of token t, for
      // channels hoff .. hoff + 31 of the half (query rows reuse the query's e^x), so both roles
      // issue 96 exponentials and 32 transposed stores per thread
      float* kbt_out = ws.kbt + (size_t)item * DK * C + t;
      auto load_x = [&](int c0, float* x) {  // gamma - rho of channels c0 .. c0 + 7
        const uint32_t g0 = grow + (uint32_t)(c0 >> 5) * 8192u;
        const float4 xa = *reinterpret_cast<const float4*>(
            sm + g0 + (((((uint32_t)c0 & 31u) >> 2) ^ tsw) << 4));
        const float4 xb = *reinterpret_cast<const float4*>(
            sm + g0 + ((((((uint32_t)c0 + 4u) & 31u) >> 2) ^ tsw) << 4));
        x[0] = xa.x; x[1] = xa.y; x[2] = xa.z; x[3] = xa.w;
        x[4] = xb.x; x[5] = xb.y; x[6] = xb.z; x[7] = xb.w;
      };
      auto load_bf8 = [&](uint32_t stg, int c0, float* y) {  // 8 staged bf16 of row t
        unpack8(*reinterpret_cast<const uint4*>(sm + stg + (uint32_t)(c0 >> 6) * 8192u + brow +
                                                 (((((uint32_t)c0 & 63u) >> 3) ^ tsw) << 4)),
                y);
      };
      auto kb_out = [&](int c0, const float* x, const float* kv, const float* er) {
        float kb[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          kb[e] = (valid ? kv[e] : 0.0f) * ex2_approx(-x[e]);
          kbt_out[(size_t)(c0 + e) * C] = kb[e] * er[e];
        }
        *reinterpret_cast<float4*>(sm + P_KB + sw128_off32(t, c0, P_KB_KB)) =
            make_float4(kb[0], kb[1], kb[2], kb[3]);
        *reinterpret_cast<float4*>(sm + P_KB + sw128_off32(t, c0 + 4, P_KB_KB)) =
            make_float4(kb[4], kb[5], kb[6], kb[7]);
      };
      if (qd < 2) {
#pragma unroll 1
        for (int cb = 0; cb < 64; cb += 16) {
          float kh[16];
#pragma unroll
          for (int u = 0; u < 16; u += 8) {
            const int c0 = chh * 64 + cb + u;
            float x[8], kv[8];
            load_x(c0, x);
            load_bf8(P_STG_K, c0, kv);
#pragma unroll
            for (int e = 0; e < 8; ++e) kh[u + e] = (valid ? kv[e] : 0.0f) * ex2_approx(x[e]);
            if ((cb & 32) == hoff) {
              const float4 ea = *reinterpret_cast<const float4*>(misc->erho + c0);
              const float4 eb = *reinterpret_cast<const float4*>(misc->erho + c0 + 4);
              const float er[8] = {ea.x, ea.y, ea.z, ea.w, eb.x, eb.y, eb.z, eb.w};
#pragma unroll
              for (int e = 0; e < 8; ++e)  // K'^T
                *f32at(sm, P_BE + sw128_off32(c0 + e, t, P_BE_KB)) = kh[u + e] * er[e];
              kb_out(c0, x, kv, er);
            }
          }
          tmem_st16(tbase + lane_base + TM_XA + chh * 64 + cb, kh);
        }
      } else {
#pragma unroll 1
        for (int cb = 0; cb < 64; cb += 16) {
          float qh[16];
#pragma unroll
          for (int u = 0; u < 16; u += 8) {
            const int c0 = chh * 64 + cb + u;
            float x[8], ex[8];
            if (need_out || (cb & 32) == hoff) {
              load_x(c0, x);
#pragma unroll
              for (int e = 0; e < 8; ++e) ex[e] = ex2_approx(x[e]);
            }
            if (need_out) {
              float qv[8];
              load_bf8(P_STG_Q, c0, qv);
#pragma unroll
              for (int e = 0; e < 8; ++e) qh[u + e] = valid ? qv[e] * ex[e] : 0.0f;
            } else {
#pragma unroll
              for (int e = 0; e < 8; ++e) qh[u + e] = 0.0f;
            }
            if ((cb & 32) == hoff) {
              float kv[8];
              load_bf8(P_STG_K, c0, kv);
              const float4 ea = *reinterpret_cast<const float4*>(misc->erho + c0);
              const float4 eb = *reinterpret_cast<const float4*>(misc->erho + c0 + 4);
              const float er[8] = {ea.x, ea.y, ea.z, ea.w, eb.x, eb.y, eb.z, eb.w};
#pragma unroll
              for (int e = 0; e < 8; ++e)  // K'^T
                *f32at(sm, P_BE + sw128_off32(c0 + e, t, P_BE_KB)) =
                    (valid ? kv[e] : 0.0f) * ex[e] * er[e];
              kb_out(c0, x, kv, er);
            }
          }
          tmem_st16(tbase + lane_base + TM_XA + chh * 64 + cb, qh);
        }
      }
    }
    if (any_strong) {
      // strong channels, rewritten by the thread that wrote them above (channels hoff ..
      // hoff + 31 of its half): no share in the A1
      // product (Kb = 0), and Kb' = k 2^(gamma_C - gamma) directly (frame 0: the staging holds
      // gamma), a factor at most 1. Kept apart so that the hot loops above carry no branch.
      const int t = (qd & 1) * 32 + lane;
      const int cw = chh * 64 + hoff;  // 32 channels, one mask word
      float* kbt_out = ws.kbt + (size_t)item * DK * C + t;
      for (uint32_t m = smask[cw >> 5]; m; m &= m - 1u) {
        const int c = cw + __ffs(m) - 1;
        const uint32_t tsw = (uint32_t)t & 7u;
        const float gam = *f32at(sm, P_STG_G + (uint32_t)(c >> 5) * 8192u + (uint32_t)t * 128u +
                                         (((((uint32_t)c & 31u) >> 2) ^ tsw) << 4) +
                                         ((uint32_t)c & 3u) * 4u);
        const float kk = t < n ? __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(
                                     sm + P_STG_K + (uint32_t)(c >> 6) * 8192u + (uint32_t)t * 128u +
                                     (((((uint32_t)c & 63u) >> 3) ^ tsw) << 4) +
                                     ((uint32_t)c & 7u) * 2u))
                               : 0.0f;
        *f32at(sm, P_KB + sw128_off32(t, c, P_KB_KB)) = 0.0f;
        kbt_out[(size_t)c * C] = kk * ex2_approx(misc->part[0][c] + misc->part[1][c] - gam);
      }
    }
    if (qd >= 2 && !((qd & 1) * 32 + lane < n)) {
      // token t past a partial chunk's end: its v row (box chh) reads as zero in the U0^T
      // product whatever the staging holds (the next range's tokens)
      if (!mbar_wait(&misc->bar_v, par)) misc->abort = 1;
      uint4* row = reinterpret_cast<uint4*>(sm + P_STG_V + chh * 8192 + ((qd & 1) * 32 + lane) * 128);
#pragma unroll
      for (int j = 0; j < 8; ++j) row[j] = make_uint4(0u, 0u, 0u, 0u);
    }
    tmem_st_wait();
    fence_proxy_async_smem();
    psync();
    // ================= A1 = [Kh; Qh] Kb^T; the staging is free: load the next item
    if (tid == 0 && !misc->abort) {
      const uint32_t ida = idesc_make(kFmtTF32, 128, 64, false, false);
      // one base descriptor per operand, advanced by constants: computing each MMA's
      // descriptor from the address would put a chain of integer ops in front of every issue
      const uint64_t dkb = sdesc_sw128(sbase + P_KB, 16, 1024);
#pragma unroll
      for (int s = 0; s < 16; ++s)
        mma_tf32_ts(tbase + TM_A1, tbase + TM_XA + s * 8,
                    desc_add(dkb, (s >> 2) * P_KB_KB + (s & 3) * 32), ida, s > 0);
      mma_commit(&misc->bar_a);
    }
    if (tid == kLoader && !misc->abort) {
      if (!any_strong) {  // else the exact strong-channel terms still read the staging
        tma_out = advance(item + stride);
        tma_par = par ^ 1u;
      }
      bulk_wait_read0();  // the previous record's W has left its staging (the solve's scratch)
      // Hand the previous item to the publishing warp: its record's store group was committed
      // a phase ago (this item's group is not committed yet), and the generic stores of its
      // record were ordered before this release by the barriers since. The publishing warp
      // stores nothing else, so its gpu-scope release does not wait on this CTA's traffic.
      if (flags && prev_item >= 0) {
        bulk_wait0();
        fence_proxy_async_global();
        hand_over(prev_item);
        prev_item = -1;
      }
    }
    if (!mbar_wait(&misc->bar_a, par)) misc->abort = 1;
    tc_fence_after();
    // Strong channels' exact shares of A_kk and A_qk, frame-free: for i <= t,
    //   sum_c k_ic (k_tc or q_tc) 2^(gamma_tc - gamma_ic),
    // every factor at most 1 (gamma is non-increasing). Rows t >= 32 against columns i < 32
    // factor through token 31 as 2^(gamma_t - gamma_31) 2^(gamma_31 - gamma_i); the second
    // factor times k_i is shared by all those rows and tabled first (at P_TBT: the previous
    // record's W left that staging before the loader's wait above). Pairs inside a diagonal
    // 32 x 32 block are taken one by one. The staging still holds this item's q, k and gamma.
    auto sg = [&](int t, int c) -> float {  // gamma_t of channel c (log2 units, frame 0)
      return *f32at(sm, P_STG_G + (uint32_t)(c >> 5) * 8192u + (uint32_t)t * 128u +
                            (((((uint32_t)c & 31u) >> 2) ^ ((uint32_t)t & 7u)) << 4) +
                            ((uint32_t)c & 3u) * 4u);
    };
    auto sbf = [&](uint32_t stg, int t, int c) -> float {  // staged bf16 of row t, channel c
      const uint32_t off = stg + (uint32_t)(c >> 6) * 8192u + (uint32_t)t * 128u +
                           (((((uint32_t)c & 63u) >> 3) ^ ((uint32_t)t & 7u)) << 4) +
                           ((uint32_t)c & 7u) * 2u;
      return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(sm + off));
    };
    float* ptab = f32at(sm, P_TBT);  // [strong channel s][32]
    if (any_strong) {
      pbar();
      int s = 0;
      for (int w4 = 0; w4 < 4; ++w4) {
        for (uint32_t m = smask[w4]; m; m &= m - 1u, ++s) {
          if ((s & 7) != warp) continue;
          const int c = w4 * 32 + __ffs(m) - 1;
          const float kj = lane < n ? sbf(P_STG_K, lane, c) : 0.0f;
          ptab[s * 32 + lane] = kj * ex2_approx(sg(31, c) - sg(lane, c));
        }
      }
      pbar();
    }
    // ================= beta_r A_kk -> scratch; TMEM A1 rows -> [0 ; tril(Aqk)]
    {
      float v[32];
      tmem_ld32(tbase + lane_base + TM_A1 + chh * 32, v);
      const int R = qd * 32 + lane;
      if (any_strong) {
        const int t = R & (C - 1), i0 = chh * 32;
        const bool qrow = R >= C;
        if (t >= i0 && (!qrow || need_out)) {  // (rows above the block are masked anyway)
          const bool diag = t < i0 + 32;     // uniform per warp, as are the other conditions
          const uint32_t stg = qrow ? P_STG_Q : P_STG_K;
          int s = 0;
          for (int w4 = 0; w4 < 4; ++w4) {
            for (uint32_t m = smask[w4]; m; m &= m - 1u, ++s) {
              const int c = w4 * 32 + __ffs(m) - 1;
              const float gt = sg(t, c);
              const float own = t < n ? sbf(stg, t, c) : 0.0f;
              if (diag) {
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                  const int i = i0 + j;
                  const float ki = i < n ? sbf(P_STG_K, i, c) : 0.0f;
                  const float f = i <= t ? ex2_approx(gt - sg(i, c)) : 0.0f;
                  v[j] = fmaf(own * ki, f, v[j]);
                }
              } else {
                const float ft = own * ex2_approx(gt - sg(31, c));
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = fmaf(ft, ptab[s * 32 + j], v[j]);
              }
            }
          }
        }
      }
      if (R < C) {
        const float br = misc->beta[R];
        float* arow = f32at(sm, SCR_A) + R * LA + chh * 32;
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
          const int i = chh * 32 + j;
          *reinterpret_cast<float4*>(arow + j) =
              make_float4(i < R ? br * v[j] : 0.0f, i + 1 < R ? br * v[j + 1] : 0.0f,
                          i + 2 < R ? br * v[j + 2] : 0.0f, i + 3 < R ? br * v[j + 3] : 0.0f);
        }
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = 0.0f;
      } else {
        const int r = R - C;
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = (chh * 32 + j <= r) ? v[j] : 0.0f;
      }
      tmem_st16(tbase + lane_base + TM_A1 + chh * 32, v);
      tmem_st16(tbase + lane_base + TM_A1 + chh * 32 + 16, v + 16);
      if (R >= C && need_out) {
        // the query rows of R start at -Q' = -Qh Diag(e^rho), so that the R product leaves
        // P K' - Q' = -Q'' / scale there (done here, where the query rows have the least work)
#pragma unroll 1
        for (int cc = chh * 64; cc < chh * 64 + 64; cc += 32) {
          float qh[32];
          tmem_ld32(tbase + lane_base + TM_XA + cc, qh);
#pragma unroll
          for (int j = 0; j < 32; j += 4) {
            const float4 e4 = *reinterpret_cast<const float4*>(misc->erho + cc + j);
            qh[j] = -qh[j] * e4.x;
            qh[j + 1] = -qh[j + 1] * e4.y;
            qh[j + 2] = -qh[j + 2] * e4.z;
            qh[j + 3] = -qh[j + 3] * e4.w;
          }
          tmem_st32(tbase + lane_base + TM_R + cc, qh);
        }
      }
      tmem_st_wait();
    }
    psync();
    if (any_strong && tid == kLoader && !misc->abort) {  // the staging is read no more
      tma_out = advance(item + stride);
      tma_par = par ^ 1u;
    }
    // ================= T = (I + A_kk)^-1 in 16 x 16 blocks
    {
      const float* Akk = f32at(sm, SCR_A);
      float* X = f32at(sm, SCR_X);
      float* Pp = f32at(sm, SCR_P);
      // diagonal blocks: lane i of a 16-lane group owns column i of its block; right-looking
      // substitution (x_l = 0 for l < i, so every update can run unconditionally)
      if (tid < 64) {
        const int blk = tid >> 4, i = tid & 15, I0 = blk * 16;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) x[r] = (r == i) ? 1.0f : 0.0f;
#pragma unroll
        for (int l = 0; l < 15; ++l)
#pragma unroll
          for (int r = l + 1; r < 16; ++r) x[r] = fmaf(-Akk[(I0 + r) * LA + I0 + l], x[l], x[r]);
#pragma unroll
        for (int r = 0; r < 16; ++r) X[(I0 + r) * LA + I0 + i] = x[r];
      } else {
        // blocks above the diagonal are zero (read by the TB pass below)
        for (int e = tid - 64; e < 6 * 256; e += kThreads - 64) {
          const int b = e >> 8, rr = (e >> 4) & 15, cc = e & 15;
          const int I = b < 3 ? 0 : (b < 5 ? 1 : 2);
          const int J = b < 3 ? b + 1 : (b < 5 ? b - 1 : 3);
          X[(I * 16 + rr) * LA + J * 16 + cc] = 0.0f;
        }
      }
      pbar();
      // Off-diagonal blocks as a 2 x 2 block inverse over 32 x 32 blocks, every 16 x 16 block
      // product a warp-level 3xTF32 MMA (fp32-level accuracy) on a 16 x 8 column half:
      //   T11 = [X00 0; X10 X11], X10 = -X11 A10 X00;  T22 = [X22 0; X32 X33], X32 = -X33 A32 X22
      //   T21 = -T22 (A21 T11)  (A21 = rows 32..63, columns 0..31 of A)
      // so the chain is four dependent products deep; the terms of A21 T11 that need only the
      // diagonal blocks run next to X10 and X32.
      const int gq = lane >> 2, tq = lane & 3;
      // d += A_IL (16 x 16 block of M, row stride LA) * B rows L*16.., columns n0 .. n0 + 7
      auto blk = [&](float* d, const float* M, int I, int L, const float* B, int bstride, int n0) {
#pragma unroll
        for (int kk = 0; kk < 16; kk += 8) {
          const float* ar = M + (I * 16 + gq) * LA + L * 16 + kk + tq;
          const float am[4] = {ar[0], ar[8 * LA], ar[4], ar[8 * LA + 4]};
          const float* br = B + (kk + tq) * bstride + n0 + gq;
          const float bv[2] = {br[0], br[4 * bstride]};
          mma16x8x8_3xtf32(d, am, bv);
        }
      };
      auto put = [&](float* dst, int stride, const float* d, float sgn) {  // 16 x 8 tile
        dst[gq * stride + 2 * tq] = sgn * d[0];
        dst[gq * stride + 2 * tq + 1] = sgn * d[1];
        dst[(gq + 8) * stride + 2 * tq] = sgn * d[2];
        dst[(gq + 8) * stride + 2 * tq + 1] = sgn * d[3];
      };
      float* Pw = Pp + warp * 128;  // this warp's [16][8] tile
      if (warp < 4) {  // X10 (warps 0, 1) and X32 (warps 2, 3), column half warp % 2
        const int J = (warp >> 1) * 2, I = J + 1, n0 = J * 16 + (warp & 1) * 8;
        float d[4] = {0.f, 0.f, 0.f, 0.f};
        blk(d, Akk, I, J, X + J * 16 * LA, LA, n0);
        put(Pw, 8, d, 1.0f);
        __syncwarp();
        float e[4] = {0.f, 0.f, 0.f, 0.f};
        blk(e, X, I, I, Pw, 8, 0);
        put(X + I * 16 * LA + n0, LA, e, -1.0f);
      } else {
        // meanwhile warps 4..7 form the terms of Y = A21 T11 that do not need X10 (the L = J
        // term of every tile of the next step), parked in T21's own blocks of X, which are
        // written only at the end
#pragma unroll 1
        for (int tt = 2 * (warp - 4); tt < 2 * (warp - 4) + 2; ++tt) {
          const int Iy = 2 + (tt >> 2), Jy = (tt >> 1) & 1, ny = Jy * 16 + (tt & 1) * 8;
          float d[4] = {0.f, 0.f, 0.f, 0.f};
          blk(d, Akk, Iy, Jy, X + Jy * 16 * LA, LA, ny);
          put(X + Iy * 16 * LA + ny, LA, d, 1.0f);
        }
      }
      pbar();
      // warp w: block (I, J) = (2 + w / 4, (w / 2) % 2) of T21, column half w % 2
      const int I2 = 2 + (warp >> 2), J2 = (warp >> 1) & 1, n2 = J2 * 16 + (warp & 1) * 8;
      {  // Y_IJ = sum_{L=J}^{1} A_IL X_LJ  (A21 T11): the L = J term is parked in X; the
         // L = 1 term of the J = 0 tiles needs X10
        const float* yp = X + I2 * 16 * LA + n2;
        float d[4] = {yp[gq * LA + 2 * tq], yp[gq * LA + 2 * tq + 1], yp[(gq + 8) * LA + 2 * tq],
                      yp[(gq + 8) * LA + 2 * tq + 1]};
        if (J2 == 0) blk(d, Akk, I2, 1, X + 16 * LA, LA, n2);
        put(Pw, 8, d, 1.0f);
      }
      pbar();
      {  // X_IJ = -sum_{L=2}^{I} X_IL Y_LJ  (Y_LJ: the tile of warp ((L - 2) << 2) | (warp & 3))
        float e[4] = {0.f, 0.f, 0.f, 0.f};
        for (int L = 2; L <= I2; ++L) blk(e, X, I2, L, Pp + (((L - 2) << 2) | (warp & 3)) * 128, 8, 0);
        put(X + I2 * 16 * LA + n2, LA, e, -1.0f);
      }
      pbar();
    }
    // ================= TB = T Diag(beta): TMEM E lanes 0..63 (lanes 64..127 zero) and TB^T
    if (qd < 2) {
      const int r = qd * 32 + lane;
      const float* xrow = f32at(sm, SCR_X) + r * LA + chh * 32;
      const float* bt = misc->beta + chh * 32;
      float v[32];
#pragma unroll
      for (int j = 0; j < 32; j += 4) {
        const float4 t4 = *reinterpret_cast<const float4*>(xrow + j);
        v[j] = t4.x * bt[j];
        v[j + 1] = t4.y * bt[j + 1];
        v[j + 2] = t4.z * bt[j + 2];
        v[j + 3] = t4.w * bt[j + 3];
      }
      tmem_st16(tbase + lane_base + TM_E + chh * 32, v);
      tmem_st16(tbase + lane_base + TM_E + chh * 32 + 16, v + 16);
      if (need_out) {  // the W rows of R start at zero (R accumulates onto all 128 rows)
        float z[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) z[j] = 0.0f;
        tmem_st32(tbase + lane_base + TM_R + chh * 64, z);
        tmem_st32(tbase + lane_base + TM_R + chh * 64 + 32, z);
      }
#pragma unroll
      for (int j = 0; j < 16; ++j)  // TB^T, first 16 of the 32 columns (the rest: warps qd >= 2)
        *f32at(sm, P_TBT + sw128_off32(chh * 32 + j, r, P_TBT_KB)) = v[j];
      // TB rows as bf16 hi and lo parts: 16-byte chunk m of the row holds columns 8 m .. 8 m + 7
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        uint32_t hw[4], lw[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float a = v[8 * m + 2 * e], b = v[8 * m + 2 * e + 1];
          const __nv_bfloat162 hi2 = __floats2bfloat162_rn(a, b);
          const __nv_bfloat162 lo2 =
              __floats2bfloat162_rn(a - __low2float(hi2), b - __high2float(hi2));
          hw[e] = *reinterpret_cast<const uint32_t*>(&hi2);
          lw[e] = *reinterpret_cast<const uint32_t*>(&lo2);
        }
        const uint32_t off =
            (uint32_t)r * 128u + ((((uint32_t)(chh * 4 + m)) ^ ((uint32_t)r & 7u)) << 4);
        *reinterpret_cast<uint4*>(sm + P_TBN + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        *reinterpret_cast<uint4*>(sm + P_TBN + 8192 + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
      }
    } else {
      float z[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) z[j] = 0.0f;
      tmem_st16(tbase + lane_base + TM_E + chh * 32, z);
      tmem_st16(tbase + lane_base + TM_E + chh * 32 + 16, z);
      {  // TB^T of row r = the thread's token, columns chh * 32 + 16 .. + 31
        const int r = (qd - 2) * 32 + lane;
        const float* xrow = f32at(sm, SCR_X) + r * LA + chh * 32 + 16;
        const float* bt = misc->beta + chh * 32 + 16;
#pragma unroll
        for (int j = 0; j < 16; j += 4) {
          const float4 t4 = *reinterpret_cast<const float4*>(xrow + j);
          const int c = chh * 32 + 16 + j;
          *f32at(sm, P_TBT + sw128_off32(c, r, P_TBT_KB)) = t4.x * bt[j];
          *f32at(sm, P_TBT + sw128_off32(c + 1, r, P_TBT_KB)) = t4.y * bt[j + 1];
          *f32at(sm, P_TBT + sw128_off32(c + 2, r, P_TBT_KB)) = t4.z * bt[j + 2];
          *f32at(sm, P_TBT + sw128_off32(c + 3, r, P_TBT_KB)) = t4.w * bt[j + 3];
        }
      }
      if (need_out) {  // tril(A_qk) rows (A1 lanes 64..127) -> row-major [t][t'] for O0^T
        const int t = (qd - 2) * 32 + lane;
        float v[32];
        tmem_ld32(tbase + lane_base + TM_A1 + chh * 32, v);
#pragma unroll
        for (int j = 0; j < 32; j += 4)
          *reinterpret_cast<float4*>(sm + P_PN + sw128_off32(t, chh * 32 + j, 8192)) =
              make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
      }
    }
    tmem_st_wait();
    fence_proxy_async_smem();
    psync();
    // ================= two independent chains of products, issued at once by two threads (one
    // thread issues an N = 64 MMA about every 50 cycles, slower than the tensor pipe runs it):
    //   thread 0:  E = [TB ; 0] + [0 ; Aqk] TB = [TB ; P], then R = [0 ; -Q'] + E K'
    //              = [W ; P K' - Q'] (with outputs; else R = E K')
    //   loader:    U0^T = V^T TB^T, then O0^T = U0^T Aqk^T
    // each product issued once its TMEM operand is complete
    if (tid == 0 && !misc->abort) {
      const uint32_t id64 = idesc_make(kFmtTF32, 128, 64, false, false);
      const uint32_t id128 = idesc_make(kFmtTF32, 128, 128, false, false);
      const uint64_t dtbt = sdesc_sw128(sbase + P_TBT, 16, 1024);
#pragma unroll
      for (int s = 0; s < 8; ++s)
        mma_tf32_ts(tbase + TM_E, tbase + TM_A1 + s * 8,
                    desc_add(dtbt, (s >> 2) * P_TBT_KB + (s & 3) * 32), id64, 1);
      mma_commit(&misc->bar_p);
      const bool ok = mbar_wait(&misc->bar_p, par);
      tc_fence_after();
      if (ok) {
        const uint64_t dbe = sdesc_sw128(sbase + P_BE, 16, 1024);
#pragma unroll
        for (int s = 0; s < 8; ++s)
          mma_tf32_ts(tbase + TM_R, tbase + TM_E + s * 8,
                      desc_add(dbe, (s >> 2) * P_BE_KB + (s & 3) * 32), id128, need_out || s > 0);
      }
      if (!ok) misc->abort = 1;
      mma_commit(&misc->bar_r);  // the record can start
    } else if (tid == kLoader && !misc->abort) {
      // U0^T = V^T (TB_hi + TB_lo)^T: A is the v staging read MN-major (value channel c of
      // token t at row t; the two 64-channel boxes 8 KiB apart), 16 tokens per K-step
      bool ok = mbar_wait(&misc->bar_v, par);
      if (ok) {
        const uint32_t idv = idesc_make(kFmtBF16, 128, 64, true, false);
        const uint64_t dv = sdesc_sw128(sbase + P_STG_V, 8192, 1024);
        const uint64_t dtbn = sdesc_sw128(sbase + P_TBN, 16, 1024);
#pragma unroll
        for (int s = 0; s < 4; ++s) {
          const uint64_t a = desc_add(dv, s * 2048);
          mma_f16(tbase + TM_U0T, a, desc_add(dtbn, s * 32), idv, s > 0);
          mma_f16(tbase + TM_U0T, a, desc_add(dtbn, 8192 + s * 32), idv, 1);
        }
      }
      mma_commit(&misc->bar_u);
      ok = ok && mbar_wait(&misc->bar_u, par);
      tc_fence_after();
      if (ok && misc->nxt[0] < n_items) {
        issue_v(misc->nxt[1], misc->nxt[3]);  // the U0^T product has read this item's v
        v_issued = true;
        v_par = par ^ 1u;
      }
      if (ok && need_out) {
        const uint32_t id64 = idesc_make(kFmtTF32, 128, 64, false, false);
        const uint64_t dpn = sdesc_sw128(sbase + P_PN, 16, 1024);
#pragma unroll
        for (int s = 0; s < 8; ++s)
          mma_tf32_ts(tbase + TM_O0T, tbase + TM_U0T + s * 8,
                      desc_add(dpn, (s >> 2) * 8192 + (s & 3) * 32), id64, s > 0);
      }
      if (!ok) misc->abort = 1;
      mma_commit(&misc->bar_e);
    }
    pbar();
    if (misc->abort) break;
    if (!mbar_wait(&misc->bar_r, par)) misc->abort = 1;
    tc_fence_after();
    // ================= workspace record: rows staged in shared memory in the boxes'
    // 128-byte swizzle (16-byte chunk j of row r at ((j ^ (r & 7)) << 4)), then bulk stores
    {
      // W (token rows 0..63) or Q'' = scale (Q' - P K') (rows 64..127): 64 columns per thread
      const int t = (qd & 1) * 32 + lane;
      if (qd < 2 || need_out) {
        const uint32_t dst = qd < 2 ? ST_W : ST_Q;
#pragma unroll 1
        for (int cc = chh * 64; cc < chh * 64 + 64; cc += 32) {
          float v[32];
          tmem_ld32(tbase + lane_base + TM_R + cc, v);
          if (qd >= 2) {  // R holds P K' - Q' there
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = -p.scale * v[j];
          }
          const uint32_t box = dst + (uint32_t)(cc >> 5) * 8192u + (uint32_t)t * 128u;
#pragma unroll
          for (int j = 0; j < 8; ++j)
            *reinterpret_cast<float4*>(sm + box + (((uint32_t)j ^ (uint32_t)(t & 7)) << 4)) =
                make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
        }
      }
      // U0^T and O0^T: value column n = TMEM lane, tokens chh * 32 .. + 31, stored straight to
      // the interleaved records (32 lanes = 32 consecutive columns = 512 contiguous bytes)
      const int nn = qd * 32 + lane;
      if (!mbar_wait(&misc->bar_u, par)) misc->abort = 1;  // long complete: O0^T came after it
      tc_fence_after();
      {
        float v[32];
        tmem_ld32(tbase + lane_base + TM_U0T + chh * 32, v);
        float4* dst = reinterpret_cast<float4*>(ws.u0 + (size_t)item * 8192) + chh * 8 * 128 + nn;
#pragma unroll
        for (int j = 0; j < 8; ++j)
          dst[j * 128] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
      }
      // O0^T, the last product
      if (!mbar_wait(&misc->bar_e, par)) misc->abort = 1;
      tc_fence_after();
      if (need_out) {
        float v[32];
        tmem_ld32(tbase + lane_base + TM_O0T + chh * 32, v);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float* w = v + 8 * k;
          uint4 pk;
          __nv_bfloat162 b0 = __floats2bfloat162_rn(p.scale * w[0], p.scale * w[1]);
          __nv_bfloat162 b1 = __floats2bfloat162_rn(p.scale * w[2], p.scale * w[3]);
          __nv_bfloat162 b2 = __floats2bfloat162_rn(p.scale * w[4], p.scale * w[5]);
          __nv_bfloat162 b3 = __floats2bfloat162_rn(p.scale * w[6], p.scale * w[7]);
          pk.x = *reinterpret_cast<uint32_t*>(&b0);
          pk.y = *reinterpret_cast<uint32_t*>(&b1);
          pk.z = *reinterpret_cast<uint32_t*>(&b2);
          pk.w = *reinterpret_cast<uint32_t*>(&b3);
          reinterpret_cast<uint4*>(ws.o0 + (size_t)item * 8192)[(chh * 4 + k) * 128 + nn] = pk;
        }
      }
    }
    fence_proxy_async_smem();
    psync();
    if (tid == kLoader) {
      if (need_out) {
#pragma unroll
        for (int kb = 0; kb < 4; ++kb)
          tma_store_2d(&twq_st, sm + ST_Q + kb * 8192, kb * 32, item * 128 + 64);
        bulk_commit();
      }
#pragma unroll
      for (int kb = 0; kb < 4; ++kb) tma_store_2d(&twq_st, sm + ST_W + kb * 8192, kb * 32, item * 128);
      bulk_commit();
      if (flags) prev_item = item;  // published during the next item's A1 product
    }
    psync();
    if (misc->abort) break;
    ++k_it;
  }
  if (misc->abort) {
    if (tid == 0 || tid == kLoader) {  // the two threads that issue MMAs
      if (tid == 0 && p.status) atomicOr(p.status, KDA_STATUS_TIMEOUT);
      mma_commit(&misc->bar_drain);
      mbar_wait(&misc->bar_drain, 0, 100000000ull);
    }
    if (tid == kLoader && tma_out) mbar_wait(&misc->bar_tma, tma_par, 100000000ull);
    if (tid == kLoader && v_issued) mbar_wait(&misc->bar_v, v_par, 100000000ull);
  }
  if (tid == kLoader) {
    bulk_wait0();
    if (flags) {  // the last item, then the end of the stream
      fence_proxy_async_global();
      if (prev_item >= 0 && !misc->abort) hand_over(prev_item);
      hand_over(-1);
    }
  }
  psync();
  if (warp == 0) tmem_dealloc(tbase, 512);
}

__global__ void __launch_bounds__(kThreads, 1)
chunk_prep_kernel(const __grid_constant__ ChunkParams p, const __grid_constant__ CUtensorMap tmq,
                  const __grid_constant__ CUtensorMap tmk,
                  const __grid_constant__ CUtensorMap tmv,
                  const __grid_constant__ CUtensorMap tmg,
                  const __grid_constant__ CUtensorMap tmb,
                  const __grid_constant__ CUtensorMap twq_st, const Ws ws, const int n_items) {
  prep_run(p, tmq, tmk, tmv, tmg, tmb, twq_st, ws, n_items, blockIdx.x, gridDim.x, nullptr);
}

// ============================================================================ kernel 2: state
// One CTA per (range, head, 128-column tile of the state): the value columns in prefill /
// replay, the M or the D half of the augmented state in package mode. The state lives in TMEM
// transposed, S^T (lane = state column n, 32-bit column = key channel c), as the A operand of
//   X^T = S^T [W ; Q'']^T   (N = 128: columns 0..63 give U^T, 64..127 the outputs)
//   Y^T = U^T Kb'           (U^T written to TMEM by the threads, N = 128 channels)
// whose B operands are the chunk's workspace rows exactly as TMA stages them. Every product is
// N = 128 wide, and nothing the threads write feeds an MMA through shared memory.
constexpr uint32_t S_STAGE = 98304;     // one chunk's [W ; Q''] (64 KiB) and Kb'^T (32 KiB)
constexpr uint32_t S_WQ = 0;            // 4 K-blocks of [128][32] fp32
constexpr uint32_t S_KBT = 65536;       // 2 K-blocks of [128][32] fp32
constexpr uint32_t S_DEC = 2 * S_STAGE;  // 3 x [128] fp32: the chunk decays (ring of 3)
constexpr uint32_t S_MISC = S_DEC + 3 * 512;
// Kept under the 196 KiB shared-memory carve-out (with the 1 KiB the system reserves per CTA),
// so that the SM keeps 60 KiB of L1 for the compute warps' U0^T / O0^T loads; at the 228 KiB
// carve-out the 28 KiB left for L1 stalled those loads for about a thousand cycles a chunk.
constexpr uint32_t S_SMEM = S_MISC + 256 + 1024;
static_assert(S_SMEM + 1024 <= 196 * 1024, "state kernel shared memory above the 196 KiB carve-out");
constexpr uint32_t TS_S = 0;     // 2 x 128: S^T, chunk j reading buffer j & 1 and writing j + 1's
constexpr uint32_t TS_X = 256;   // 128: X^T
constexpr uint32_t TS_U = 384;   // 64: U^T
// 8 compute warps + 1 MMA-issuing warp + 1 warp that loads the records + 2 warps that drop
// consumed records from L2 (fused launch). Twelve warps cost no registers over nine: either way
// three share an SMSP's register file.
constexpr int kStateThreads = kThreads + 128;

struct StateMisc {
  uint64_t full[2];     // TMA: chunk j's record landed in stage j & 1 (and decay slot j % 3)
  uint64_t s_ready;     // compute warps: the initial S^T written
  uint64_t r_ready;     // compute warps: S^T Diag(e^gamma_C) written into the next buffer
  uint64_t u_ready[2];  // compute warps: U^T tokens 32 h .. 32 h + 31 written
  uint64_t x_free;      // compute warps: done reading X^T
  uint64_t empty[2];    // MMAs: stage s read by its chunk's products (the next load may come)
  uint64_t bar_x, bar_y, bar_drain;
  uint32_t tmem_base;
  int abort;
  uint32_t consumed;  // compute-warp arrivals: 8 per chunk whose record they are done with
};
static_assert(sizeof(StateMisc) <= 256, "misc overflow");

// Compute warp w (0..7): TMEM lane quarter w % 4, so state column n = 32 (w % 4) + lane of the
// tile; half h = w / 4 of the channels (state update) and of the tokens (U and outputs). Warp 8
// issues the MMAs, warp 10 the records' TMA loads (two chunks ahead, each stage refilled once
// the products have read it); they and the compute warps synchronise through mbarriers only.
// With p.discard, warps 9 and 11 drop each chunk's record from L2 once the compute warps have
// counted it consumed.
// With `flags`, waits (acquire) for each item's record before reading it.
// The walk of range ridx for (tile, head), in TMEM the caller allocated; ends on a CTA barrier
// (the caller then reads misc->abort). The barriers are initialised afresh for each range.
// kDeferOut: store a chunk's outputs during the next chunk's X product (the standalone walk,
// which reads its records from memory: ~15% faster on a 256-chunk walk) or at once (the fused
// launch, where the walk trails the prep CTAs and storing at once measured better). A template
// parameter, so that each kernel carries one form and no registers for the other.
// kMultiRange: the CTA walks further ranges after this one in TMEM the caller allocated, so
// every asynchronous arrive on the barriers is waited for before they are initialised again;
// otherwise the walk allocates and frees its TMEM itself.
template <bool kDeferOut, bool kMultiRange>
__device__ __forceinline__ void state_range(const ChunkParams& p, const CUtensorMap& twq,
                                            const CUtensorMap& tkbt, const CUtensorMap& tdec,
                                            const Ws& ws, const int tile, const int h,
                                            const int ridx, const uint32_t* flags) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  StateMisc* misc = reinterpret_cast<StateMisc*>(sm + S_MISC);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool issuer = warp == 8;
  const bool discarder = warp == 9 || warp == 11;
  const bool loader = warp == 10;
  const int qd = warp & 3, hf = (warp >> 2) & 1;
  const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
  const int H = p.H;
  const bool pkg = p.package != 0;
  const bool mcols = pkg && tile == 0;      // package mode: tile 0 = M, tile 1 = D
  const int n = qd * 32 + lane;              // state column of this thread within the tile

  int t_begin = 0, t_end = p.total_tokens;
  if (p.offsets) {
    t_begin = p.offsets[ridx];
    t_end = p.offsets[ridx + 1];
    if (t_end < t_begin || t_begin < 0 || t_end > p.total_tokens) {
      if (tid == 0 && p.status) atomicOr(p.status, KDA_STATUS_BAD_OFFSETS);
      t_end = t_begin;
    }
  }
  const int nch = (t_end - t_begin + C - 1) / C;
  const int slot0 = t_begin / C + ridx;

  if (!kMultiRange && warp == 0) {
    tmem_alloc(&misc->tmem_base, 512);
    tmem_relinquish();
  }
  if (tid == 0) {  // (with kMultiRange every async arrive of the previous range has landed)
    if (!kMultiRange) misc->abort = 0;
    mbar_init(&misc->full[0], 1);
    mbar_init(&misc->full[1], 1);
    mbar_init(&misc->s_ready, 8);
    mbar_init(&misc->r_ready, 8);
    mbar_init(&misc->u_ready[0], 4);
    mbar_init(&misc->u_ready[1], 4);
    mbar_init(&misc->x_free, 8);
    mbar_init(&misc->empty[0], 1);
    mbar_init(&misc->empty[1], 1);
    mbar_init(&misc->bar_x, 1);
    mbar_init(&misc->bar_y, 1);
    mbar_init(&misc->bar_drain, 1);
    misc->consumed = 0;
    fence_mbar_init();
  }
  cta_sync();
  const uint32_t tbase = misc->tmem_base;
  const uint32_t sbase = smem_u32(sm);

  if (issuer) {
    // ------------------------------------------------------------ MMA-issuing warp (lane 0)
    if (lane == 0) {
      const uint32_t idesc = idesc_make(kFmtTF32, 128, 128, false, false);
      const uint32_t idesc_x = pkg ? idesc_make(kFmtTF32, 128, 64, false, false) : idesc;
      bool ok = true;
      for (int j = 0; j < nch && ok; ++j) {
        const uint32_t par = (uint32_t)j & 1u;
        const uint32_t st = (uint32_t)(j & 1) * S_STAGE;
        const uint64_t d_wq = sdesc_sw128(sbase + st + S_WQ, 16, 1024);
        const uint64_t d_kbt = sdesc_sw128(sbase + st + S_KBT, 16, 1024);
        const uint32_t s_cur = tbase + TS_S + par * 128u, s_nxt = tbase + TS_S + (par ^ 1u) * 128u;
        ok = mbar_wait_or(&misc->full[j & 1], ((uint32_t)j >> 1) & 1u, &misc->abort);
        // X^T = S_j^T [W ; Q'']^T once S_j is complete (the initial state, or the previous
        // chunk's Y product) and the compute warps are done with the previous X^T
        if (j == 0) {
          ok = ok && mbar_wait_or(&misc->s_ready, 0, &misc->abort);
        } else {
          ok = ok && mbar_wait_or(&misc->bar_y, par ^ 1u, &misc->abort) &&
               mbar_wait_or(&misc->x_free, par ^ 1u, &misc->abort);
        }
        tc_fence_after();
        if (!ok) break;
#pragma unroll
        for (int ks = 0; ks < 16; ++ks)  // K-step: channels 8 ks .. 8 ks + 7
          mma_tf32_ts(tbase + TS_X, s_cur + ks * 8,
                      desc_add(d_wq, (ks >> 2) * 16384 + (ks & 3) * 32), idesc_x, ks > 0);
        mma_commit(&misc->bar_x);
        // S_{j+1}^T = S_j^T Diag(e^gamma_C) + U^T Kb': accumulated onto the decayed state that
        // the compute warps wrote into the other buffer, token half by token half as U^T is
        // written
        ok = mbar_wait_or(&misc->r_ready, par, &misc->abort);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          ok = ok && mbar_wait_or(&misc->u_ready[hh], par, &misc->abort);
          tc_fence_after();
          if (ok) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int ks = hh * 4 + k;  // K-step: tokens 8 ks .. 8 ks + 7
              mma_tf32_ts(s_nxt, tbase + TS_U + ks * 8,
                          desc_add(d_kbt, (ks >> 2) * 16384 + (ks & 3) * 32), idesc, 1);
            }
          }
        }
        if (!ok) break;
        mma_commit(&misc->bar_y);
        mma_commit(&misc->empty[j & 1]);  // both products have read the stage
      }
      if (!ok) {
        misc->abort = 1;
        mma_commit(&misc->bar_drain);
        mbar_wait(&misc->bar_drain, 0, 100000000ull);
      } else if (kMultiRange) {  // the last two stage releases have arrived
        for (int j = nch > 2 ? nch - 2 : 0; j < nch; ++j)
          mbar_wait(&misc->empty[j & 1], ((uint32_t)j >> 1) & 1u, 100000000ull);
      }
    }
  } else if (loader) {
    // ------------------------------------------------------------ loading warp (lane 0)
    // Chunk j's record into stage j & 1 (and decay slot j % 3), two chunks ahead: chunk j + 2
    // as soon as chunk j's products have read the stage. Kept off the MMA-issuing thread, whose
    // chain the stage's release, a record's flag and the copies' issue would otherwise lengthen.
    if (lane == 0) {
      tma_prefetch_desc(&twq);
      tma_prefetch_desc(&tkbt);
      tma_prefetch_desc(&tdec);
      auto issue_tma = [&](int j) -> bool {
        const int item = (slot0 + j) * H + h;
        if (flags) {  // the record is published by the prep CTA that wrote it
          if (!wait_flag(flags + item, p.flag_wait_ns)) return false;
          fence_proxy_async_global();
        }
        uint8_t* st = sm + (j & 1) * S_STAGE;
        uint64_t* bar = &misc->full[j & 1];
        // package mode has no outputs: the boxes hold W's 64 rows only (not Q'')
        mbar_arrive_expect_tx(bar, (pkg ? 32768u : 65536u) + 32768u + 512u);
#pragma unroll
        for (int kb = 0; kb < 4; ++kb)
          tma_load_2d(st + S_WQ + kb * 16384, &twq, bar, kb * 32, item * 128);
#pragma unroll
        for (int kb = 0; kb < 2; ++kb)
          tma_load_2d(st + S_KBT + kb * 16384, &tkbt, bar, kb * 32, item * 128);
        tma_load_2d(sm + S_DEC + (j % 3) * 512, &tdec, bar, 0, item);
        // the compute warps read this chunk's U0^T / O0^T rows with plain loads one chunk
        // ahead; bring them into L2 now
        if (!mcols) bulk_prefetch_l2(ws.u0 + (int64_t)item * 8192, 32768);
        if (!pkg) bulk_prefetch_l2(ws.o0 + (int64_t)item * 8192, 16384);
        return true;
      };
      int tma_last = -1;
      bool ok = true;
      for (int j = 0; j < nch && ok; ++j) {
        if (j >= 2) ok = mbar_wait_or(&misc->empty[j & 1], ((uint32_t)(j - 2) >> 1) & 1u, &misc->abort);
        ok = ok && issue_tma(j);
        if (ok) tma_last = j;
      }
      if (!ok) {
        misc->abort = 1;
        // this warp's copies in flight land before the CTA lets go of its shared memory
        for (int j = tma_last > 0 ? tma_last - 1 : 0; j <= tma_last; ++j)
          mbar_wait(&misc->full[j & 1], ((uint32_t)j >> 1) & 1u, 100000000ull);
      }
    }
  } else if (discarder) {
    // ------------------------------------------------------------ discarding warps
    // The records of a fused launch are read once, from L2: drop each chunk's lines once the
    // compute warps are done with it (both products complete, U0^T / O0^T in registers), so
    // that they are never written back to DRAM. A discard holds its thread for ~100 cycles, so
    // they run here, off the compute warps' chain, in two warps (one takes every record's first
    // 578 lines, the other the rest: one warp fell behind the walk); a warp more than two
    // chunks behind skips ahead (a skipped record is merely written back).
    if (p.discard) {
      const int l0 = warp == 9 ? 0 : 578, l1 = warp == 9 ? 578 : 1156;
      for (int j = 0; j < nch; ++j) {
        const uint64_t t0 = globaltimer_ns();
        uint32_t c;
        while ((c = ld_acquire_cta(&misc->consumed)) < 8u * (uint32_t)(j + 1)) {  // bounded
          if (*(volatile int*)&misc->abort) break;
          if (globaltimer_ns() - t0 > 4000000000ull) {
            misc->abort = 1;
            break;
          }
          __nanosleep(64);
        }
        if (*(volatile int*)&misc->abort) break;
        const int behind = (int)(c >> 3) - (j + 1);
        if (behind > 2) j += behind - 2;
        const int64_t item = (int64_t)(slot0 + j) * H + h;
        const uint8_t* r_wq = reinterpret_cast<const uint8_t*>(ws.wq + item * 128 * 128);
        const uint8_t* r_kb = reinterpret_cast<const uint8_t*>(ws.kbt + item * 128 * 64);
        const uint8_t* r_u0 = reinterpret_cast<const uint8_t*>(ws.u0 + item * 8192);
        const uint8_t* r_o0 = reinterpret_cast<const uint8_t*>(ws.o0 + item * 8192);
        const uint8_t* r_dc = reinterpret_cast<const uint8_t*>(ws.dec + item * 128);
        // 512 lines of [W ; Q''], 256 of Kb'^T, 256 of U0^T, 128 of O0^T, 4 of the decays
        for (int l = l0 + lane; l < l1; l += 32) {
          const uint8_t* a = l < 512    ? r_wq + l * 128
                             : l < 768  ? r_kb + (l - 512) * 128
                             : l < 1024 ? r_u0 + (l - 768) * 128
                             : l < 1152 ? r_o0 + (l - 1024) * 128
                                        : r_dc + (l - 1152) * 128;
          discard_l2_line(a);
        }
      }
    }
  } else {
    // ------------------------------------------------------------ compute warps
    const int64_t sh = (int64_t)ridx * H + h;
    const int vcol = pkg ? (mcols ? -1 : n) : n;  // value column of U0 / outputs (-1: none)
    {  // S^T rows n, channels 64 hf .. 64 hf + 63
      float v[32];
#pragma unroll 1
      for (int cc = hf * 64; cc < hf * 64 + 64; cc += 32) {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int c = cc + i;
          float x = 0.0f;
          if (pkg) x = (mcols && c == n) ? 1.0f : 0.0f;
          else if (p.init) x = p.init[(sh * DK + c) * DK + n];
          v[i] = x;
        }
        tmem_st32(tbase + lane_base + TS_S + cc, v);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&misc->s_ready);
    }
    // per-chunk register operands, loaded one chunk ahead: U0^T[n][32 hf ..] (32 fp32) and
    // O0^T[n][32 hf ..] (32 bf16)
    // U0^T first (needed by the U step), O0^T second (needed by the outputs), each issued as
    // soon as the previous chunk's registers are consumed
    auto load_u0 = [&](int j, float4* u0) {
      const int64_t item = (int64_t)(slot0 + j) * H + h;
      if (flags) {
        // The loading warp acquired the record's flag before its arrive on this chunk's stage
        // barrier (a release): acquiring that phase orders these loads after the record.
        if (!mbar_wait_or(&misc->full[j & 1], ((uint32_t)j >> 1) & 1u, &misc->abort))
          misc->abort = 1;
      }
      if (vcol >= 0) {
        const float4* src = reinterpret_cast<const float4*>(ws.u0 + item * 8192) + hf * 8 * 128 + vcol;
#pragma unroll
        for (int i = 0; i < 8; ++i) u0[i] = __ldg(src + i * 128);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) u0[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    };
    auto load_o0 = [&](int j, uint4* o0) {  // after load_u0 of the same chunk (its acquire)
      const int64_t item = (int64_t)(slot0 + j) * H + h;
      if (!pkg) {
        const uint4* src = reinterpret_cast<const uint4*>(ws.o0 + item * 8192) + hf * 4 * 128 + n;
#pragma unroll
        for (int i = 0; i < 4; ++i) o0[i] = __ldg(src + i * 128);
      }
    };
    float4 u0[8];
    uint4 o0[4];
#pragma unroll
    for (int i = 0; i < 8; ++i) u0[i] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < 4; ++i) o0[i] = make_uint4(0, 0, 0, 0);
    if (nch > 0) {
      load_u0(0, u0);
      load_o0(0, o0);
    }
    // A chunk's outputs (bf16 pairs of adjacent tokens of column n): token t of column n, 32
    // lanes = 64 contiguous bytes of one token's row; none once the CTA gave up. Lanes l and
    // l ^ 1 trade halves so that the even lane holds columns (n, n + 1) of the even tokens and
    // the odd lane those of the odd tokens: 16 four-byte stores per thread.
    uint32_t ob16[16];
    int prev_t0 = 0, prev_nvalid = 0;
    auto store_out = [&](int ot0, int onvalid) {
      if (!pkg && p.o && !misc->abort) {
        const bool odd = (lane & 1) != 0;
        __nv_bfloat16* o = (__nv_bfloat16*)p.o + ((int64_t)ot0 * H + h) * DK + (n & ~1);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const uint32_t mine = ob16[i];  // (token 2i, token 2i + 1) of column n
          const uint32_t give = odd ? (mine & 0xFFFFu) : (mine >> 16);
          const uint32_t got = __shfl_xor_sync(0xFFFFFFFFu, give, 1);
          const uint32_t pair = odd ? (got | (mine & 0xFFFF0000u)) : ((mine & 0xFFFFu) | (got << 16));
          const int t = hf * 32 + 2 * i + (odd ? 1 : 0);
          if (t < onvalid) *reinterpret_cast<uint32_t*>(o + (int64_t)t * H * DK) = pair;
        }
      }
    };

    for (int j = 0; j < nch; ++j) {
      const int t0 = t_begin + j * C;
      const int nvalid = min(C, t_end - t0);
      const uint32_t par = (uint32_t)j & 1u;
      const uint32_t s_cur = tbase + lane_base + TS_S + par * 128u;
      const uint32_t s_nxt = tbase + lane_base + TS_S + (par ^ 1u) * 128u;
      // ================= S_j^T Diag(e^gamma_C) into the other buffer (channels 64 hf ..), while
      // the X product reads S_j^T; the Y product then accumulates onto it. S_j^T is complete
      // with the previous chunk's Y product; the decays came with this chunk's record.
      if (j > 0 && !mbar_wait_relaxed_or(&misc->bar_y, par ^ 1u, &misc->abort)) misc->abort = 1;
      if (!mbar_wait_or(&misc->full[j & 1], ((uint32_t)j >> 1) & 1u, &misc->abort))
        misc->abort = 1;
      tc_fence_after();
      {
        // the thread's 64 channels in four loads of 16 columns, all in flight at once
        const float* dec = f32at(sm, S_DEC + (j % 3) * 512);
        const int c0 = hf * 64;
        uint32_t sr[4][16];
#pragma unroll
        for (int k = 0; k < 4; ++k) tmem_ld16_nowait(s_cur + c0 + 16 * k, sr[k]);
        tmem_ld_wait();
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int cc = c0 + 16 * k;
          float sd[16];
#pragma unroll
          for (int i = 0; i < 16; i += 4) {
            const float4 d4 = *reinterpret_cast<const float4*>(dec + cc + i);
            sd[i] = d4.x * __uint_as_float(sr[k][i]);
            sd[i + 1] = d4.y * __uint_as_float(sr[k][i + 1]);
            sd[i + 2] = d4.z * __uint_as_float(sr[k][i + 2]);
            sd[i + 3] = d4.w * __uint_as_float(sr[k][i + 3]);
          }
          tmem_st16(s_nxt + cc, sd);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_relaxed(&misc->r_ready);
      }
      // the previous chunk's outputs, while the X product runs
      if (kDeferOut && j > 0) store_out(prev_t0, prev_nvalid);
      // ================= U^T = U0^T - (W S)^T (tokens 32 hf ..), then the output values
      if (!mbar_wait_relaxed_or(&misc->bar_x, par, &misc->abort)) misc->abort = 1;
      tc_fence_after();
      {
        float x[32];
        tmem_ld32(tbase + lane_base + TS_X + hf * 32, x);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          x[4 * i] = u0[i].x - x[4 * i];
          x[4 * i + 1] = u0[i].y - x[4 * i + 1];
          x[4 * i + 2] = u0[i].z - x[4 * i + 2];
          x[4 * i + 3] = u0[i].w - x[4 * i + 3];
        }
        tmem_st32(tbase + lane_base + TS_U + hf * 32, x);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_relaxed(&misc->u_ready[hf]);
      }
      if (j + 1 < nch) load_u0(j + 1, u0);  // this chunk's U0^T is consumed
      // output values of tokens 32 hf .. 32 hf + 31: O^T[n][t] = (Q'' S)^T + O0^T, packed as
      // bf16 pairs of adjacent tokens, stored during the next chunk's X product
      if (!pkg && p.o) {
        float x[32];
        tmem_ld32(tbase + lane_base + TS_X + 64 + hf * 32, x);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          float ob[8];
          unpack8(o0[k], ob);
#pragma unroll
          for (int e = 0; e < 8; e += 2) {
            __nv_bfloat162 b = __floats2bfloat162_rn(x[8 * k + e] + ob[e], x[8 * k + e + 1] + ob[e + 1]);
            ob16[4 * k + e / 2] = *reinterpret_cast<uint32_t*>(&b);
          }
        }
      }
      tc_fence_before();  // this warp is done with X^T
      __syncwarp();
      if (lane == 0) mbar_arrive_relaxed(&misc->x_free);
      if (j + 1 < nch) load_o0(j + 1, o0);  // this chunk's O0^T is consumed
      if (kDeferOut) {
        prev_t0 = t0;
        prev_nvalid = nvalid;
      } else {
        store_out(t0, nvalid);
      }
      if (p.discard) {
        // the chunk's record is read no more (its tensor copies landed, U0^T / O0^T used):
        // count it consumed for the discarding warp (release: the warp's loads came first)
        __syncwarp();
        if (lane == 0) {
          __threadfence_block();
          atomicAdd(&misc->consumed, 1u);
        }
      }
      if (misc->abort) break;
    }
    if (kDeferOut && nch > 0) store_out(prev_t0, prev_nvalid);  // the last chunk's outputs
  }
  cta_sync();
  if (!issuer && !discarder && !loader && !misc->abort) {  // exit state rows c of column n
    const int64_t sh = (int64_t)ridx * H + h;
    float* dst = nullptr;
    if (pkg) dst = mcols ? p.M + sh * DK * DK + n : p.D + sh * DK * DK + n;
    else if (p.final_state) dst = p.final_state + sh * DK * DK + n;
    // the final state is in buffer nch & 1, complete with the last Y product (waited for even
    // when not stored if a further range re-initialises the barrier)
    if ((dst || kMultiRange) && nch > 0 &&
        !mbar_wait_relaxed_or(&misc->bar_y, (uint32_t)(nch - 1) & 1u, &misc->abort))
      dst = nullptr;
    tc_fence_after();
    if (dst) {
#pragma unroll 1
      for (int cc = hf * 64; cc < hf * 64 + 64; cc += 32) {
        float s[32];
        tmem_ld32(tbase + lane_base + TS_S + (uint32_t)(nch & 1) * 128u + cc, s);
#pragma unroll
        for (int i = 0; i < 32; ++i) dst[(int64_t)(cc + i) * DK] = s[i];
      }
    }
  }
  if (!kMultiRange) {
    if (misc->abort && tid == 0 && p.status) atomicOr(p.status, KDA_STATUS_TIMEOUT);
    cta_sync();
    if (warp == 0) tmem_dealloc(tbase, 512);
  } else {
    cta_sync();
  }
}

// TMEM for a walk CTA: allocated once (all 512 columns), released at the end.
__device__ __forceinline__ void state_tmem_alloc() {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  StateMisc* misc = reinterpret_cast<StateMisc*>(sm + S_MISC);
  if ((threadIdx.x >> 5) == 0) {
    tmem_alloc(&misc->tmem_base, 512);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) misc->abort = 0;
}
__device__ __forceinline__ void state_tmem_free(const ChunkParams& p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  StateMisc* misc = reinterpret_cast<StateMisc*>(sm + S_MISC);
  if (misc->abort && threadIdx.x == 0 && p.status) atomicOr(p.status, KDA_STATUS_TIMEOUT);
  cta_sync();
  if ((threadIdx.x >> 5) == 0) tmem_dealloc(misc->tmem_base, 512);
}

__global__ void __launch_bounds__(kStateThreads, 1)
chunk_state_kernel(const __grid_constant__ ChunkParams p,
                   const __grid_constant__ CUtensorMap twq,
                   const __grid_constant__ CUtensorMap tkbt,
                   const __grid_constant__ CUtensorMap tdec, const Ws ws,
                   const uint32_t* flags) {
  state_range<true, false>(p, twq, tkbt, tdec, ws, blockIdx.x, blockIdx.y, blockIdx.z, flags);
}

// ============================================================================ fused launch
// One cooperative launch of exactly one CTA per SM for inputs with few (range, head) pairs:
// CTAs 0 .. n_state - 1 run the state kernel's work for (tile, head, range), the others the
// prep kernel's items; a state CTA reads an item's record once its prep CTA has published it
// (flags[item] = 1, release / acquire at gpu scope; every wait bounded). The serial state
// walk then follows the parallel prep work instead of waiting for all of it.
constexpr uint32_t F_SMEM = P_SMEM > S_SMEM ? P_SMEM : S_SMEM;
constexpr int kFusedMaxRanges = 8;  // ranges one walk CTA may take in turn

// kLooped: a walk CTA takes ranges_per_walk ranges in turn; else exactly one (ranges_per_walk
// is 1), walked as in the state kernel (a separate instance, so that the one-range launch
// carries none of the multi-range bookkeeping).
template <bool kLooped>
__global__ void __launch_bounds__(kStateThreads, 1)
chunk_fused_kernel(const __grid_constant__ ChunkParams p, const __grid_constant__ CUtensorMap tmq,
                   const __grid_constant__ CUtensorMap tmk,
                   const __grid_constant__ CUtensorMap tmv,
                   const __grid_constant__ CUtensorMap tmg,
                   const __grid_constant__ CUtensorMap tmb,
                   const __grid_constant__ CUtensorMap twq_st,
                   const __grid_constant__ CUtensorMap twq,
                   const __grid_constant__ CUtensorMap tkbt,
                   const __grid_constant__ CUtensorMap tdec, const Ws ws, const int n_items,
                   const int n_state, const int ranges_per_walk, uint32_t* flags) {
  const int b = blockIdx.x;
  if (b < n_state) {
    // walk CTA b: (tile, head) b % (tiles H), ranges_per_walk consecutive ranges
    const int tiles = p.package ? 2 : 1;
    const int r0 = b / (tiles * p.H) * ranges_per_walk;
    const int r1 = min(r0 + ranges_per_walk, p.n_ranges);
    if (kLooped) {
      extern __shared__ uint8_t smem_raw[];
      uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
      const StateMisc* misc = reinterpret_cast<const StateMisc*>(sm + S_MISC);
      state_tmem_alloc();
      for (int r = r0; r < r1; ++r) {
        state_range<false, true>(p, twq, tkbt, tdec, ws, b % tiles, (b / tiles) % p.H, r, flags);
        if (misc->abort) break;  // read after the range's closing CTA barrier: uniform
      }
      state_tmem_free(p);
    } else if (r0 < r1) {
      state_range<false, false>(p, twq, tkbt, tdec, ws, b % tiles, (b / tiles) % p.H, r0, flags);
    }
  } else {
    // the prep work uses 8 warps; the ninth publishes the finished items' flags (the others,
    // which load and discard records in the state CTAs, have nothing to do here)
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    PrepMisc* misc = reinterpret_cast<PrepMisc*>(sm + P_MISC);
    if (threadIdx.x == 0) misc->pub_head = misc->pub_tail = 0;
    __syncthreads();
    if (threadIdx.x < kThreads) {
      prep_run(p, tmq, tmk, tmv, tmg, tmb, twq_st, ws, n_items, b - n_state,
               (int)gridDim.x - n_state, flags);
    } else if (threadIdx.x == kThreads) {
      for (uint32_t c = 0;; ++c) {
        // bounded: the loader hands over an item per prep iteration, and ends the stream
        const uint64_t t0 = globaltimer_ns();
        bool got = true;
        while (ld_acquire_cta(&misc->pub_head) <= c) {
          if (globaltimer_ns() - t0 > 4000000000ull) { got = false; break; }
          __nanosleep(32);
        }
        if (!got) break;
        const int item = misc->pub_ring[c & 3];
        if (item < 0) break;
        st_release_gpu(flags + item, 1u);
        st_release_cta(&misc->pub_tail, c + 1);
      }
    }
  }
}

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (EncodeTiledFn)f;
  }
  return fn;
}

// [T, H, 128] (bf16, or fp32 when f32) viewed as a 3-D tensor (128, H, T); box (box_d, 1, 64)
// with the 128-byte swizzle.
bool make_map3(CUtensorMap* m, const void* ptr, int T, int H, int box_d, bool f32) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t es_bytes = f32 ? 4 : 2;
  cuuint64_t dims[3] = {(cuuint64_t)DK, (cuuint64_t)H, (cuuint64_t)(T > 0 ? T : 1)};
  cuuint64_t strides[2] = {(cuuint64_t)DK * es_bytes, (cuuint64_t)H * DK * es_bytes};
  cuuint32_t box[3] = {(cuuint32_t)box_d, 1, (cuuint32_t)C};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                   const_cast<void*>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// beta [T, H] fp32 as a 2-D tensor (H, T); box (4 heads, 64 tokens).
bool make_map_beta(CUtensorMap* m, const float* ptr, int T, int H) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)H, (cuuint64_t)(T > 0 ? T : 1)};
  cuuint64_t strides[1] = {(cuuint64_t)H * 4};
  cuuint32_t box[2] = {4, (cuuint32_t)C};
  cuuint32_t es[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(ptr), dims, strides,
                   box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// [rows][cols] workspace array (fp32, or bf16 when bf16) as a 2-D tensor (cols, rows); box of
// 128 bytes x box_rows with the 128-byte swizzle: one K-block of an operand per copy.
bool make_map_ws(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows,
                 bool bf16 = false) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const uint64_t es_bytes = bf16 ? 2 : 4;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(cols * es_bytes)};
  cuuint32_t box[2] = {(cuuint32_t)(128 / es_bytes), box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
                   const_cast<void*>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// dec [items][128] fp32 as a 2-D tensor (128, items); box (128, 1): one item's decays.
bool make_map_dec(CUtensorMap* m, const float* ptr, uint64_t items) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)DK, (cuuint64_t)items};
  cuuint64_t strides[1] = {(cuuint64_t)DK * 4};
  cuuint32_t box[2] = {(cuuint32_t)DK, 1};
  cuuint32_t es[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(ptr), dims, strides,
                   box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int64_t n_items_of(int n_ranges, int total_tokens, int H) {
  return ((int64_t)total_tokens / C + n_ranges) * H;
}

bool cooperative_ok() {
  int dev = 0, v = 0;
  return cudaGetDevice(&dev) == cudaSuccess &&
         cudaDeviceGetAttribute(&v, cudaDevAttrCooperativeLaunch, dev) == cudaSuccess && v != 0;
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    n = 148;
  return n;
}

}  // namespace

bool chunk_tc_shape_ok(kda_dtype dt, int n_ranges, int total_tokens, int H, int dk, int dv) {
  return dt == KDA_BF16 && dk == 128 && dv == 128 && total_tokens > 0 && H % 4 == 0 &&
         n_items_of(n_ranges, total_tokens, H) * 128 < ((int64_t)1 << 31);
}

size_t chunk_tc_workspace_bytes(int n_ranges, int total_tokens, int H) {
  const size_t items = (size_t)n_items_of(n_ranges, total_tokens, H);
  return items * kItemBytes + ((items * 4 + 255) & ~(size_t)255);  // records, then flags
}

bool chunk_tc_available() { return encode_fn() != nullptr; }

bool make_map_rows(CUtensorMap* m, const void* ptr, bool f32, uint64_t cols, uint64_t rows,
                   uint32_t box_cols, uint32_t box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const uint64_t es = f32 ? 4 : 2;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)(rows > 0 ? rows : 1)};
  cuuint64_t strides[1] = {(cuuint64_t)(cols * es)};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                   const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

kda_status launch_chunk_tc(const ChunkParams& p, kda_dtype dt, void* workspace, size_t ws_bytes,
                           cudaStream_t s, int phases) {
  (void)dt;
  if (p.n_ranges == 0) return KDA_OK;
  const int64_t n_items = n_items_of(p.n_ranges, p.total_tokens, p.H);
  const size_t need = chunk_tc_workspace_bytes(p.n_ranges, p.total_tokens, p.H);
  if (!workspace || ws_bytes < need || ((uintptr_t)workspace % 256) != 0)
    return set_error(KDA_ERR_WORKSPACE, "tensor-core chunk path: workspace too small");
  uint8_t* base = (uint8_t*)workspace;
  Ws ws;
  ws.wq = (float*)base;
  ws.kbt = (float*)(base + (size_t)n_items * kWqBytes);
  ws.u0 = (float*)(base + (size_t)n_items * (kWqBytes + kKbtBytes));
  ws.o0 = (__nv_bfloat16*)(base + (size_t)n_items * (kWqBytes + kKbtBytes + kU0Bytes));
  ws.dec = (float*)(base + (size_t)n_items * (kWqBytes + kKbtBytes + kU0Bytes + kO0Bytes));
  uint32_t* flags = (uint32_t*)(base + (size_t)n_items * kItemBytes);

  const bool do_prep = (phases & kPhasePrep) != 0, do_state = (phases & kPhaseState) != 0;
  ChunkParams pp = p;
  if (pp.flag_wait_ns == 0) pp.flag_wait_ns = 4000000000ull;
  pp.discard = 0;
  CUtensorMap mq, mk, mv, mg, mb, mwq, mkbt, mdec, swq;
  const uint64_t rows128 = (uint64_t)n_items * 128;
  bool maps_ok = true;
  if (do_prep) {
    const void* qp = p.q ? p.q : p.k;
    maps_ok = make_map3(&mq, qp, p.total_tokens, p.H, 64, false) &&
              make_map3(&mk, p.k, p.total_tokens, p.H, 64, false) &&
              make_map3(&mv, p.v, p.total_tokens, p.H, 64, false) &&
              make_map3(&mg, p.g, p.total_tokens, p.H, 32, true) &&
              make_map_beta(&mb, p.beta, p.total_tokens, p.H) &&
              make_map_ws(&swq, ws.wq, rows128, 128, 64);
  }
  if (maps_ok && do_state) {
    maps_ok = make_map_ws(&mwq, ws.wq, rows128, 128, p.package ? 64 : 128) &&
              make_map_ws(&mkbt, ws.kbt, rows128, 64, 128) &&
              make_map_dec(&mdec, ws.dec, (uint64_t)n_items);
  }
  if (!maps_ok)
    return set_error(KDA_ERR_CUDA, "tensor-core chunk path: cuTensorMapEncodeTiled failed");
  cudaError_t e =
      cudaFuncSetAttribute(chunk_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, P_SMEM);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(chunk_state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             S_SMEM);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(chunk_fused_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             F_SMEM);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(chunk_fused_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             F_SMEM);
  if (e != cudaSuccess)
    return set_error(KDA_ERR_CUDA, std::string("tensor-core chunk path attribute: ") +
                                       cudaGetErrorString(e));
  const int tiles = p.package ? 2 : 1;
  const int sms = sm_count();
  // Few serial walks: run them next to the prep work in one cooperative launch (at most a
  // quarter of the SMs walk, the rest prepare records). Every (tile, head, range) its own walk
  // CTA when they fit; else, for a few ranges (a few long sequences, whose serial walks would
  // otherwise follow all of the prep work), one walk CTA per (tile, head) takes the ranges in
  // order while the prep CTAs produce their records in that order.
  const int64_t per_range = (int64_t)tiles * p.H;
  int ranges_per_walk = 0;
  if (per_range * p.n_ranges * 4 <= sms) ranges_per_walk = 1;
  else if (p.n_ranges <= kFusedMaxRanges && per_range * 4 <= sms) ranges_per_walk = p.n_ranges;
  const int64_t n_state =
      ranges_per_walk ? per_range * ((p.n_ranges + ranges_per_walk - 1) / ranges_per_walk) : 0;
  if (do_prep && do_state && ranges_per_walk > 0 && cooperative_ok()) {
    e = cudaMemsetAsync(flags, 0, (size_t)n_items * 4, s);
    if (e != cudaSuccess)
      return set_error(KDA_ERR_CUDA, std::string("tensor-core chunk path flags: ") +
                                         cudaGetErrorString(e));
    // the fused launch owns its records and its walks read them while they are still in L2:
    // the walk drops each one once read (one reader per record: not in package mode, where the
    // M and D tiles read the same one; with two launches the records have long left L2)
    ChunkParams pf = pp;
    pf.discard = p.package ? 0 : 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)sms);
    cfg.blockDim = dim3(kStateThreads);
    cfg.dynamicSmemBytes = F_SMEM;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = ranges_per_walk > 1
            ? cudaLaunchKernelEx(&cfg, chunk_fused_kernel<true>, pf, mq, mk, mv, mg, mb, swq, mwq,
                                 mkbt, mdec, ws, (int)n_items, (int)n_state, ranges_per_walk, flags)
            : cudaLaunchKernelEx(&cfg, chunk_fused_kernel<false>, pf, mq, mk, mv, mg, mb, swq, mwq,
                                 mkbt, mdec, ws, (int)n_items, (int)n_state, ranges_per_walk, flags);
    if (e == cudaSuccess) {
      count_launches(1);
      return check_launch("tensor-core chunk fused kernel");
    }
    (void)cudaGetLastError();  // not co-resident here: two launches instead
  }
  if (do_prep) {
    const int grid1 = (int)std::min<int64_t>(n_items, sms);
    chunk_prep_kernel<<<grid1, kThreads, P_SMEM, s>>>(pp, mq, mk, mv, mg, mb, swq, ws,
                                                       (int)n_items);
    count_launches(1);
    kda_status st = check_launch("tensor-core chunk prep kernel");
    if (st != KDA_OK || !do_state) return st;
  }
  dim3 grid2(tiles, p.H, p.n_ranges);
  chunk_state_kernel<<<grid2, kStateThreads, S_SMEM, s>>>(
      pp, mwq, mkbt, mdec, ws, (phases & kPhaseFlags) ? flags : nullptr);
  count_launches(1);
  return check_launch("tensor-core chunk state kernel");
}

}  // namespace kda
