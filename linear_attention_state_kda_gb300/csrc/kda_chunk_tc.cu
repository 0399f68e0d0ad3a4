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
// where Kh = k e^(gamma - rho), Qh = q e^(gamma - rho), Kb = k e^(rho - gamma) and
// rho = gamma_C / 2: in this midpoint frame every factor stays within e^(+-80) as long as a
// chunk decays by at most 160 nats per channel (beyond it KDA_STATUS_DECAY_RANGE is raised).
//
// Kernel 1 (prep) computes the state-independent factors of every (chunk, head) in parallel
// (persistent CTAs, one item at a time, the next item's loads in flight) and writes them to a
// workspace record. Kernel 2 (state) walks each range's chunks in order for one (range, head,
// 32-column tile of the state): per chunk one MMA for [W; Q''] S, the U update on CUDA cores,
// one MMA for Kb'^T U, and the state update, with the records streamed in by TMA two chunks
// ahead. In package mode kernel 2 runs the same chunks on a 32-column tile of the augmented
// state [M | D] (identity / zero start; M columns see zero values) and writes no outputs.
//
// All MMAs are kind::tf32 with fp32 accumulation; every shared-memory operand is K-major in
// the 128-byte swizzle, and operands needed in the other orientation are written transposed
// by the threads that produce them or staged in TMEM. Waits on mbarriers are bounded (2 s of
// globaltimer); on expiry a CTA raises KDA_STATUS_TIMEOUT, drains its own MMAs and copies
// (bounded), frees its TMEM and returns.
#include <cuda.h>

#include <algorithm>

#include "kda_internal.cuh"
#include "ptx.cuh"

namespace kda {
namespace {

using namespace ptx;

constexpr int C = kChunk;  // 64 tokens per chunk
constexpr int DK = 128;
constexpr int TW = 32;     // state columns per state-kernel CTA
constexpr int kThreads = 256;
constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------- workspace record
// Per item (chunk slot, head):
//   wq  [128][128] fp32  rows 0..63 W, rows 64..127 Q''
//   kbt [128][64]  fp32  Kb'^T
//   u0  [64][128]  fp32  U0
//   o0  [64][128]  bf16  O0
//   dec [128]      fp32  e^gamma_C
// Chunk j of range i (starting at token b_i) has slot floor(b_i / C) + i + j: distinct for
// distinct chunks of valid ordered ranges, and below floor(T / C) + n_ranges.
constexpr size_t kWqBytes = 128 * 128 * 4;
constexpr size_t kKbtBytes = 128 * 64 * 4;
constexpr size_t kU0Bytes = 64 * 128 * 4;
constexpr size_t kO0Bytes = 64 * 128 * 2;
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
constexpr uint32_t P_BE = P_KB + 32768;  // [K'^T ; V^T] [256][64 tok] fp32 (2 K-blocks)
constexpr uint32_t P_BE_KB = 32768;
constexpr uint32_t P_TBT = P_BE + 65536;  // TB^T [64][64] fp32 (2 K-blocks of 8 KiB)
constexpr uint32_t P_TBT_KB = 8192;
constexpr uint32_t P_XTRA = P_TBT + 16384;
constexpr int LA = 68;                    // padded row length of the solve scratch
constexpr uint32_t SCR_A = P_KB;          // beta_r A_kk [64][68] (Kb is dead by then)
constexpr uint32_t SCR_X = P_XTRA;        // (I + A_kk)^-1 [64][68]
constexpr uint32_t SCR_P = P_XTRA + 64 * LA * 4;  // 8 warps x [16][8]
constexpr uint32_t P_MISC = SCR_P + 8 * 128 * 4;
// Workspace-record staging for the bulk-tensor stores, over Kb, [K'^T ; V^T] and TB^T (all
// dead once R is complete): W, Q'' and U0 as 4 boxes of [64 rows][32] fp32, O0 as 2 boxes of
// [64 rows][64] bf16, each in the 128-byte swizzle.
constexpr uint32_t ST_W = P_KB;
constexpr uint32_t ST_Q = P_KB + 32768;
constexpr uint32_t ST_U = P_KB + 65536;
constexpr uint32_t ST_O = P_KB + 98304;
static_assert(ST_O + 16384 <= P_XTRA, "record staging overflow");
constexpr uint32_t P_SMEM = P_MISC + 2048 + 1024;
static_assert(64 * LA * 4 <= 32768, "A_kk scratch must fit in the Kb buffer");
static_assert(P_KB % 1024 == 0 && P_BE % 1024 == 0 && P_TBT % 1024 == 0, "alignment");

// TMEM columns (512)
constexpr uint32_t TM_XA = 0;    // 128: [Kh ; Qh] (lanes = tokens), the A operand of A1
constexpr uint32_t TM_A1 = 128;  // 64: [Kh ; Qh] Kb^T -> [0 ; Aqk], the A operand of P
constexpr uint32_t TM_E = 192;   // 64: [TB ; 0] + [0 ; Aqk] TB = [TB ; P], the A operand of E
constexpr uint32_t TM_R = 256;   // 256: [TB ; P] [K' | V] = [W | U0 ; P K' | P V]

struct PrepMisc {
  uint64_t bar_tma, bar_a, bar_p, bar_e, bar_drain;
  uint32_t tmem_base;
  int abort;
  int nxt[4];  // item, t0, n, head of the item whose loads are in flight
  float part[2][DK];
  float erho[DK];
  float beta[C];
};
static_assert(sizeof(PrepMisc) <= 2048, "misc overflow");

__global__ void __launch_bounds__(kThreads, 1)
chunk_prep_kernel(const __grid_constant__ ChunkParams p, const __grid_constant__ CUtensorMap tmq,
                  const __grid_constant__ CUtensorMap tmk,
                  const __grid_constant__ CUtensorMap tmv,
                  const __grid_constant__ CUtensorMap tmg,
                  const __grid_constant__ CUtensorMap tmb,
                  const __grid_constant__ CUtensorMap twq_st,
                  const __grid_constant__ CUtensorMap tu0_st,
                  const __grid_constant__ CUtensorMap to0_st, const Ws ws, const int n_items) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  PrepMisc* misc = reinterpret_cast<PrepMisc*>(sm + P_MISC);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int qd = warp & 3;    // TMEM lane quarter
  const int chh = warp >> 2;  // half of the columns / channels
  const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
  const bool need_out = p.package == 0;
  const uint32_t tx_bytes = (need_out ? 16384u : 0u) + 16384u + 16384u + 32768u + 1024u;

  if (warp == 0) {
    tmem_alloc(&misc->tmem_base, 512);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(&misc->bar_tma, 1);
    mbar_init(&misc->bar_a, 1);
    mbar_init(&misc->bar_p, 1);
    mbar_init(&misc->bar_e, 1);
    mbar_init(&misc->bar_drain, 1);
    misc->abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmk);
    tma_prefetch_desc(&tmv);
    tma_prefetch_desc(&tmg);
    tma_prefetch_desc(&tmb);
    if (need_out) tma_prefetch_desc(&tmq);
  }
  cta_sync();
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
    tma_load_3d(sm + P_STG_V, &tmv, &misc->bar_tma, 0, hh, t0);
    tma_load_3d(sm + P_STG_V + 8192, &tmv, &misc->bar_tma, 64, hh, t0);
#pragma unroll
    for (int kb = 0; kb < 4; ++kb)
      tma_load_3d(sm + P_STG_G + kb * 8192, &tmg, &misc->bar_tma, kb * 32, hh, t0);
    tma_load_2d(sm + P_STG_B, &tmb, &misc->bar_tma, hh & ~3, t0);
  };
  // thread 0: finds this CTA's next item holding a chunk, from `from` on, and issues its loads
  auto advance = [&](int from) {
    int it = from, t0 = 0, n = 0, hh = 0;
    while (it < n_items && !item_chunk(p, it, t0, n, hh)) it += gridDim.x;
    misc->nxt[0] = it;
    misc->nxt[1] = t0;
    misc->nxt[2] = n;
    misc->nxt[3] = hh;
    if (it < n_items) issue_tma(t0, hh);
    return it < n_items;
  };
  // Loads are issued by the loader thread (warp 1), MMAs by thread 0, so that the next item's
  // loads go out while thread 0 is issuing the A1 product.
  constexpr int kLoader = 32;
  bool tma_out = false;  // loader: a load is in flight, completing phase parity tma_par
  uint32_t tma_par = 0;
  if (tid == kLoader) tma_out = advance(blockIdx.x);
  cta_sync();

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
      __syncthreads();
      const float p0 = misc->part[0][c], p1 = misc->part[1][c];
      const float rho2 = 0.5f * (p0 + p1);  // log2 units
      if (half == 0) {
        misc->erho[c] = ex2_approx(rho2);
        ws.dec[(size_t)item * DK + c] = ex2_approx(p0 + p1);
        if (!((p0 + p1) >= -kMaxChunkDecay * kLog2e) && p.status)
          atomicOr(p.status, KDA_STATUS_DECAY_RANGE);
      }
      // gamma - rho (log2 units) in place of g: each element has one owner
      float gam = half ? p0 : 0.0f;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        gam += gl[i];
        *f32at(sm, gbase + (uint32_t)i * 128u + ((xg ^ (uint32_t)(i & 7)) << 4)) = gam - rho2;
      }
    }
    if (tid == 0) bulk_wait_read0();  // the previous record has left the staging buffers
    __syncthreads();
    // ================= operands (row role: token t; key rows in warps 0,1,4,5, query rows
    // and values in warps 2,3,6,7; channel half chh)
    {
      const int t = (qd & 1) * 32 + lane;
      const bool valid = t < n;
      const uint32_t tsw = (uint32_t)(t & 7);
      const uint32_t grow = P_STG_G + (uint32_t)t * 128u;
      const uint32_t brow = (uint32_t)t * 128u;
      // Kb (the B operand of A1) and Kb'^T (workspace) of token t: key-row threads cover the
      // first 32 channels of their half, query-row threads the last 32, so both roles issue
      // 96 exponentials per thread
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
      auto kb_out = [&](int c0, const float* x, const float* kv) {
        float kb[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          kb[e] = (valid ? kv[e] : 0.0f) * ex2_approx(-x[e]);
          kbt_out[(size_t)(c0 + e) * C] = kb[e] * misc->erho[c0 + e];
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
            for (int e = 0; e < 8; ++e) {
              kh[u + e] = (valid ? kv[e] : 0.0f) * ex2_approx(x[e]);
              *f32at(sm, P_BE + sw128_off32(c0 + e, t, P_BE_KB)) =
                  kh[u + e] * misc->erho[c0 + e];  // K'^T
            }
            if (cb < 32) kb_out(c0, x, kv);
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
            float vv[8], x[8];
            load_bf8(P_STG_V, c0, vv);
#pragma unroll
            for (int e = 0; e < 8; ++e)
              *f32at(sm, P_BE + sw128_off32(128 + c0 + e, t, P_BE_KB)) = valid ? vv[e] : 0.0f;
            if (need_out || cb >= 32) load_x(c0, x);
            if (need_out) {
              float qv[8];
              load_bf8(P_STG_Q, c0, qv);
#pragma unroll
              for (int e = 0; e < 8; ++e) qh[u + e] = valid ? qv[e] * ex2_approx(x[e]) : 0.0f;
            } else {
#pragma unroll
              for (int e = 0; e < 8; ++e) qh[u + e] = 0.0f;
            }
            if (cb >= 32) {
              float kv[8];
              load_bf8(P_STG_K, c0, kv);
              kb_out(c0, x, kv);
            }
          }
          tmem_st16(tbase + lane_base + TM_XA + chh * 64 + cb, qh);
        }
      }
    }
    tmem_st_wait();
    fence_proxy_async_smem();
    cta_sync();
    // ================= A1 = [Kh; Qh] Kb^T; the staging is free: load the next item
    if (tid == 0 && !misc->abort) {
      const uint32_t ida = idesc_make(kFmtTF32, 128, 64, false, false);
#pragma unroll
      for (int s = 0; s < 16; ++s) {
        const uint64_t b =
            sdesc_sw128(sbase + P_KB + (s >> 2) * P_KB_KB + (s & 3) * 32, 16, 1024);
        mma_tf32_ts(tbase + TM_A1, tbase + TM_XA + s * 8, b, ida, s > 0);
      }
      mma_commit(&misc->bar_a);
    }
    if (tid == kLoader && !misc->abort) {
      tma_out = advance(item + gridDim.x);
      tma_par = par ^ 1u;
    }
    if (!mbar_wait(&misc->bar_a, par)) misc->abort = 1;
    tc_fence_after();
    // ================= beta_r A_kk -> scratch; TMEM A1 rows -> [0 ; tril(Aqk)]
    {
      float v[32];
      tmem_ld32(tbase + lane_base + TM_A1 + chh * 32, v);
      const int R = qd * 32 + lane;
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
      tmem_st_wait();
    }
    cta_sync();
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
      __syncthreads();
      // off-diagonal blocks by distance d: X_IJ = -X_II sum_{L=J}^{I-1} A_IL X_LJ (J = I - d).
      // Warp w < 2 (4 - d) owns block J = w / 2 and its 8-column half w % 2; both 16 x 16
      // block products run as warp-level 3xTF32 MMAs (fp32-level accuracy), the partial
      // product passing through a per-warp 16 x 8 tile of shared memory.
      const int gq = lane >> 2, tq = lane & 3;
      float* Pw = Pp + warp * 128;  // [16][8]
      for (int dist = 1; dist < 4; ++dist) {
        if (warp < 2 * (4 - dist)) {
          const int J = warp >> 1, I = J + dist, n0 = J * 16 + (warp & 1) * 8;
          float d[4] = {0.f, 0.f, 0.f, 0.f};
          for (int L = J; L < I; ++L) {
#pragma unroll
            for (int kk = 0; kk < 16; kk += 8) {
              const float* ar = Akk + (I * 16 + gq) * LA + L * 16 + kk + tq;
              const float a[4] = {ar[0], ar[8 * LA], ar[4], ar[8 * LA + 4]};
              const float* br = X + (L * 16 + kk + tq) * LA + n0 + gq;
              const float bv[2] = {br[0], br[4 * LA]};
              mma16x8x8_3xtf32(d, a, bv);
            }
          }
          Pw[gq * 8 + 2 * tq] = d[0];
          Pw[gq * 8 + 2 * tq + 1] = d[1];
          Pw[(gq + 8) * 8 + 2 * tq] = d[2];
          Pw[(gq + 8) * 8 + 2 * tq + 1] = d[3];
          __syncwarp();
          float e[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int kk = 0; kk < 16; kk += 8) {
            const float* ar = X + (I * 16 + gq) * LA + I * 16 + kk + tq;
            const float a[4] = {ar[0], ar[8 * LA], ar[4], ar[8 * LA + 4]};
            const float bv[2] = {Pw[(kk + tq) * 8 + gq], Pw[(kk + tq + 4) * 8 + gq]};
            mma16x8x8_3xtf32(e, a, bv);
          }
          float* xr = X + (I * 16 + gq) * LA + n0 + 2 * tq;
          xr[0] = -e[0];
          xr[1] = -e[1];
          xr[8 * LA] = -e[2];
          xr[8 * LA + 1] = -e[3];
          __syncwarp();
        }
        __syncthreads();
      }
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
#pragma unroll
      for (int j = 0; j < 32; ++j)
        *f32at(sm, P_TBT + sw128_off32(chh * 32 + j, r, P_TBT_KB)) = v[j];
    } else {
      float z[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) z[j] = 0.0f;
      tmem_st16(tbase + lane_base + TM_E + chh * 32, z);
      tmem_st16(tbase + lane_base + TM_E + chh * 32 + 16, z);
    }
    tmem_st_wait();
    fence_proxy_async_smem();
    cta_sync();
    // ================= E = [TB ; 0] + [0 ; Aqk] TB, then R = E [K' | V]
    if (tid == 0 && !misc->abort) {
      const uint32_t idp = idesc_make(kFmtTF32, 128, 64, false, false);
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        const uint64_t b =
            sdesc_sw128(sbase + P_TBT + (s >> 2) * P_TBT_KB + (s & 3) * 32, 16, 1024);
        mma_tf32_ts(tbase + TM_E, tbase + TM_A1 + s * 8, b, idp, 1);
      }
      mma_commit(&misc->bar_p);
      if (!mbar_wait(&misc->bar_p, par)) {
        misc->abort = 1;
      } else {
        tc_fence_after();
        const uint32_t ide = idesc_make(kFmtTF32, 128, 256, false, false);
#pragma unroll
        for (int s = 0; s < 8; ++s) {
          const uint64_t b =
              sdesc_sw128(sbase + P_BE + (s >> 2) * P_BE_KB + (s & 3) * 32, 16, 1024);
          mma_tf32_ts(tbase + TM_R, tbase + TM_E + s * 8, b, ide, s > 0);
        }
        mma_commit(&misc->bar_e);
      }
    }
    __syncthreads();
    if (misc->abort) break;
    if (!mbar_wait(&misc->bar_e, par)) misc->abort = 1;
    tc_fence_after();
    // ================= workspace record: rows staged in shared memory in the boxes'
    // 128-byte swizzle (16-byte chunk j of row t at ((j ^ (t & 7)) << 4)), then bulk stores
    {
      const int t = (qd & 1) * 32 + lane;
      const uint32_t rsw = (uint32_t)t * 128u;
      const uint32_t tx = (uint32_t)(t & 7);
      if (qd < 2 || (need_out && chh == 0)) {  // fp32 rows: W, U0 or Q'' = scale (Q' - P K')
        const uint32_t dst = qd < 2 ? (chh == 0 ? ST_W : ST_U) : ST_Q;
        const uint32_t src = qd < 2 ? TM_R + chh * 128 : TM_R;
#pragma unroll 1
        for (int cc = 0; cc < 128; cc += 32) {
          float v[32];
          tmem_ld32(tbase + lane_base + src + cc, v);
          if (qd >= 2) {
            float qh[32];
            tmem_ld32(tbase + lane_base + TM_XA + cc, qh);
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = p.scale * (qh[j] * misc->erho[cc + j] - v[j]);
          }
          const uint32_t box = dst + (uint32_t)(cc >> 5) * 8192u + rsw;
#pragma unroll
          for (int j = 0; j < 8; ++j)
            *reinterpret_cast<float4*>(sm + box + (((uint32_t)j ^ tx) << 4)) =
                make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
        }
      } else if (need_out) {  // O0 = scale P V (bf16)
#pragma unroll 1
        for (int cc = 0; cc < 128; cc += 32) {
          float v[32];
          tmem_ld32(tbase + lane_base + TM_R + 128 + cc, v);
          const uint32_t box = ST_O + (uint32_t)(cc >> 6) * 8192u + rsw;
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
            const uint32_t jc = (uint32_t)((cc & 63) >> 3) + (uint32_t)k;
            *reinterpret_cast<uint4*>(sm + box + ((jc ^ tx) << 4)) = pk;
          }
        }
      }
    }
    fence_proxy_async_smem();
    cta_sync();
    if (tid == 0) {
#pragma unroll
      for (int kb = 0; kb < 4; ++kb) {
        tma_store_2d(&twq_st, sm + ST_W + kb * 8192, kb * 32, item * 128);
        tma_store_2d(&tu0_st, sm + ST_U + kb * 8192, kb * 32, item * 64);
        if (need_out) tma_store_2d(&twq_st, sm + ST_Q + kb * 8192, kb * 32, item * 128 + 64);
      }
      if (need_out) {
        tma_store_2d(&to0_st, sm + ST_O, 0, item * 64);
        tma_store_2d(&to0_st, sm + ST_O + 8192, 64, item * 64);
      }
      bulk_commit();
    }
    cta_sync();
    if (misc->abort) break;
    ++k_it;
  }
  if (misc->abort) {
    if (tid == 0) {
      if (p.status) atomicOr(p.status, KDA_STATUS_TIMEOUT);
      mma_commit(&misc->bar_drain);
      mbar_wait(&misc->bar_drain, 0, 100000000ull);
    }
    if (tid == kLoader && tma_out) mbar_wait(&misc->bar_tma, tma_par, 100000000ull);
  }
  if (tid == 0) bulk_wait0();
  cta_sync();
  if (warp == 0) tmem_dealloc(tbase, 512);
}

// ============================================================================ kernel 2: state
constexpr uint32_t S_STAGE = 98304;     // one chunk's [W ; Q''] (64 KiB) and Kb'^T (32 KiB)
constexpr uint32_t S_WQ = 0;            // 4 K-blocks of [128][32] fp32
constexpr uint32_t S_KBT = 65536;       // 2 K-blocks of [128][32] fp32
constexpr uint32_t S_SH = 2 * S_STAGE;  // S^T [32 cols][128 ch] fp32 (4 K-blocks of 4 KiB)
constexpr uint32_t S_UT = S_SH + 16384;  // U^T [32 cols][64 tok] fp32 (2 K-blocks of 4 KiB)
constexpr uint32_t S_MISC = S_UT + 8192;
constexpr uint32_t S_SMEM = S_MISC + 128 + 1024;
constexpr uint32_t TS_X = 0;   // 32 columns: [W ; Q''] S
constexpr uint32_t TS_Y = 32;  // 32 columns: Kb'^T U

struct StateMisc {
  uint64_t full[2], bar_x, bar_y, bar_drain;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(StateMisc) <= 128, "misc overflow");

__global__ void __launch_bounds__(kThreads, 1)
chunk_state_kernel(const __grid_constant__ ChunkParams p,
                   const __grid_constant__ CUtensorMap twq,
                   const __grid_constant__ CUtensorMap tkbt, const Ws ws) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  StateMisc* misc = reinterpret_cast<StateMisc*>(sm + S_MISC);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int qd = warp & 3, chh = warp >> 2;
  const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
  const int tile = blockIdx.x, h = blockIdx.y, ridx = blockIdx.z;
  const int H = p.H;
  const bool pkg = p.package != 0;
  const int j0 = tile * TW;
  const bool mcols = pkg && j0 < DK;
  const int vcol0 = pkg ? j0 - DK : j0;
  const int c = qd * 32 + lane;  // state row (key channel); token row of U (c < 64) / O (c - 64)
  const int col0 = chh * 16;     // 16 of the tile's columns

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

  if (warp == 0) {
    tmem_alloc(&misc->tmem_base, 64);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(&misc->full[0], 1);
    mbar_init(&misc->full[1], 1);
    mbar_init(&misc->bar_x, 1);
    mbar_init(&misc->bar_y, 1);
    mbar_init(&misc->bar_drain, 1);
    misc->abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&twq);
    tma_prefetch_desc(&tkbt);
  }
  // state tile in registers: row c, columns col0 .. col0 + 15
  float s[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int col = col0 + j;
    float x = 0.0f;
    if (pkg) x = (mcols && c == j0 + col) ? 1.0f : 0.0f;
    else if (p.init) x = p.init[(((int64_t)ridx * H + h) * DK + c) * DK + j0 + col];
    s[j] = x;
  }
  auto store_sh = [&]() {  // S^T as the K-major B operand: element (row = column, k = c)
#pragma unroll
    for (int j = 0; j < 16; ++j) *f32at(sm, S_SH + sw128_off32(col0 + j, c, 4096)) = s[j];
  };
  store_sh();
  fence_proxy_async_smem();
  cta_sync();
  const uint32_t tbase = misc->tmem_base;
  const uint32_t sbase = smem_u32(sm);

  auto issue_tma = [&](int j) {  // chunk j into stage j & 1
    const int item = (slot0 + j) * H + h;
    uint8_t* st = sm + (j & 1) * S_STAGE;
    uint64_t* bar = &misc->full[j & 1];
    mbar_arrive_expect_tx(bar, S_STAGE);
#pragma unroll
    for (int kb = 0; kb < 4; ++kb)
      tma_load_2d(st + S_WQ + kb * 16384, &twq, bar, kb * 32, item * 128);
#pragma unroll
    for (int kb = 0; kb < 2; ++kb)
      tma_load_2d(st + S_KBT + kb * 16384, &tkbt, bar, kb * 32, item * 128);
  };
  int tma_last = -1;  // thread 0: last chunk whose loads were issued
  if (tid == 0) {
    for (int j = 0; j < 2 && j < nch; ++j) {
      issue_tma(j);
      tma_last = j;
    }
  }
  // per-chunk register operands (prefetched one chunk ahead)
  auto load_regs = [&](int j, float* u0, uint4* o0, float& dec) {
    const int64_t item = (int64_t)(slot0 + j) * H + h;
    dec = __ldg(ws.dec + item * DK + c);
    if (qd < 2) {
      if (!mcols) {
        const float4* src =
            reinterpret_cast<const float4*>(ws.u0 + (item * 64 + c) * 128 + vcol0 + col0);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float4 t4 = __ldg(src + i);
          u0[4 * i] = t4.x;
          u0[4 * i + 1] = t4.y;
          u0[4 * i + 2] = t4.z;
          u0[4 * i + 3] = t4.w;
        }
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) u0[i] = 0.0f;
      }
    } else if (!pkg) {
      const uint4* src =
          reinterpret_cast<const uint4*>(ws.o0 + (item * 64 + (c - 64)) * 128 + j0 + col0);
      o0[0] = __ldg(src);
      o0[1] = __ldg(src + 1);
    }
  };
  float u0[16], nu0[16], dec = 0.0f, ndec = 0.0f;
  uint4 o0[2], no0[2];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    u0[i] = 0.0f;
    nu0[i] = 0.0f;
  }
  o0[0] = o0[1] = no0[0] = no0[1] = make_uint4(0, 0, 0, 0);
  if (nch > 0) load_regs(0, u0, o0, dec);
  __syncthreads();

  bool ok = true;
  for (int j = 0; j < nch; ++j) {
    const int t0 = t_begin + j * C;
    const int n = min(C, t_end - t0);
    const uint32_t par = (uint32_t)j & 1u;
    const uint32_t st = (uint32_t)(j & 1) * S_STAGE;
    // ================= X = [W ; Q''] S
    if (tid == 0) {
      if (!mbar_wait(&misc->full[j & 1], ((uint32_t)j >> 1) & 1u)) {
        misc->abort = 1;
      } else {
        tc_fence_after();
        const uint32_t idx = idesc_make(kFmtTF32, 128, 32, false, false);
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const uint64_t a =
              sdesc_sw128(sbase + st + S_WQ + (k >> 2) * 16384 + (k & 3) * 32, 16, 1024);
          const uint64_t b = sdesc_sw128(sbase + S_SH + (k >> 2) * 4096 + (k & 3) * 32, 16, 1024);
          mma_tf32(tbase + TS_X, a, b, idx, k > 0);
        }
        mma_commit(&misc->bar_x);
      }
    }
    if (j + 1 < nch) load_regs(j + 1, nu0, no0, ndec);  // next chunk's register operands
    if (!mbar_wait(&misc->bar_x, par)) misc->abort = 1;
    tc_fence_after();
    // ================= U = U0 - W S (token rows), kept as U^T for the next product
    float x[16];
    tmem_ld16(tbase + lane_base + TS_X + col0, x);
    if (qd < 2) {
#pragma unroll
      for (int i = 0; i < 16; ++i)
        *f32at(sm, S_UT + sw128_off32(col0 + i, c, 4096)) = u0[i] - x[i];
    }
    fence_proxy_async_smem();
    cta_sync();
    if (misc->abort) {
      ok = false;
      break;
    }
    // ================= Y = Kb'^T U; outputs O = Q'' S + O0 meanwhile
    if (tid == 0) {
      const uint32_t idy = idesc_make(kFmtTF32, 128, 32, false, false);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint64_t a =
            sdesc_sw128(sbase + st + S_KBT + (k >> 2) * 16384 + (k & 3) * 32, 16, 1024);
        const uint64_t b = sdesc_sw128(sbase + S_UT + (k >> 2) * 4096 + (k & 3) * 32, 16, 1024);
        mma_tf32(tbase + TS_Y, a, b, idy, k > 0);
      }
      mma_commit(&misc->bar_y);
    }
    if (qd >= 2 && !pkg && p.o) {
      const int r = c - 64;
      if (r < n) {
        __nv_bfloat16* o = (__nv_bfloat16*)p.o + ((int64_t)(t0 + r) * H + h) * DK + j0 + col0;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          float ob[8];
          unpack8(o0[hh], ob);
          const float* xx = x + 8 * hh;
          uint4 pk;
          __nv_bfloat162 b0 = __floats2bfloat162_rn(xx[0] + ob[0], xx[1] + ob[1]);
          __nv_bfloat162 b1 = __floats2bfloat162_rn(xx[2] + ob[2], xx[3] + ob[3]);
          __nv_bfloat162 b2 = __floats2bfloat162_rn(xx[4] + ob[4], xx[5] + ob[5]);
          __nv_bfloat162 b3 = __floats2bfloat162_rn(xx[6] + ob[6], xx[7] + ob[7]);
          pk.x = *reinterpret_cast<uint32_t*>(&b0);
          pk.y = *reinterpret_cast<uint32_t*>(&b1);
          pk.z = *reinterpret_cast<uint32_t*>(&b2);
          pk.w = *reinterpret_cast<uint32_t*>(&b3);
          *reinterpret_cast<uint4*>(o + 8 * hh) = pk;
        }
      }
    }
    if (!mbar_wait(&misc->bar_y, par)) misc->abort = 1;
    tc_fence_after();
    // ================= S = Diag(e^gamma_C) S + Y; this chunk's stage is free
    if (tid == 0 && j + 2 < nch && !misc->abort) {
      issue_tma(j + 2);
      tma_last = j + 2;
    }
    {
      float y[16];
      tmem_ld16(tbase + lane_base + TS_Y + col0, y);
#pragma unroll
      for (int i = 0; i < 16; ++i) s[i] = fmaf(dec, s[i], y[i]);
      store_sh();
    }
    fence_proxy_async_smem();
    cta_sync();
    if (misc->abort) {
      ok = false;
      break;
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) u0[i] = nu0[i];
    o0[0] = no0[0];
    o0[1] = no0[1];
    dec = ndec;
  }
  if (misc->abort) ok = false;
  if (!ok) {
    if (tid == 0) {
      if (p.status) atomicOr(p.status, KDA_STATUS_TIMEOUT);
      mma_commit(&misc->bar_drain);
      mbar_wait(&misc->bar_drain, 0, 100000000ull);
      // the last two issued loads are the only ones that can still be in flight
      for (int j = tma_last > 0 ? tma_last - 1 : 0; j <= tma_last; ++j)
        mbar_wait(&misc->full[j & 1], ((uint32_t)j >> 1) & 1u, 100000000ull);
    }
  } else {
    const int64_t sh = (int64_t)ridx * H + h;
    float* dst = nullptr;
    if (pkg) dst = mcols ? p.M + (sh * DK + c) * DK + j0 : p.D + (sh * DK + c) * DK + vcol0;
    else if (p.final_state) dst = p.final_state + (sh * DK + c) * DK + j0;
    if (dst) {
#pragma unroll
      for (int j = 0; j < 16; j += 4)
        *reinterpret_cast<float4*>(dst + col0 + j) =
            make_float4(s[j], s[j + 1], s[j + 2], s[j + 3]);
    }
  }
  cta_sync();
  if (warp == 0) tmem_dealloc(tbase, 64);
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

int64_t n_items_of(int n_ranges, int total_tokens, int H) {
  return ((int64_t)total_tokens / C + n_ranges) * H;
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
  return (size_t)n_items_of(n_ranges, total_tokens, H) * kItemBytes;
}

bool chunk_tc_supported(const ChunkParams& p, kda_dtype dt) {
  return chunk_tc_shape_ok(dt, p.n_ranges, p.total_tokens, p.H, p.dk, p.dv) &&
         ((uintptr_t)p.beta % 16) == 0 && encode_fn() != nullptr;
}

kda_status launch_chunk_tc(const ChunkParams& p, kda_dtype dt, void* workspace, size_t ws_bytes,
                           cudaStream_t s) {
  (void)dt;
  if (p.n_ranges == 0) return KDA_OK;
  const int64_t n_items = n_items_of(p.n_ranges, p.total_tokens, p.H);
  const size_t need = (size_t)n_items * kItemBytes;
  if (!workspace || ws_bytes < need || ((uintptr_t)workspace % 256) != 0)
    return set_error(KDA_ERR_WORKSPACE, "tensor-core chunk path: workspace too small");
  uint8_t* base = (uint8_t*)workspace;
  Ws ws;
  ws.wq = (float*)base;
  ws.kbt = (float*)(base + (size_t)n_items * kWqBytes);
  ws.u0 = (float*)(base + (size_t)n_items * (kWqBytes + kKbtBytes));
  ws.o0 = (__nv_bfloat16*)(base + (size_t)n_items * (kWqBytes + kKbtBytes + kU0Bytes));
  ws.dec = (float*)(base + (size_t)n_items * (kWqBytes + kKbtBytes + kU0Bytes + kO0Bytes));

  CUtensorMap mq, mk, mv, mg, mb, mwq, mkbt, swq, su0, so0;
  const void* qp = p.q ? p.q : p.k;
  const uint64_t rows128 = (uint64_t)n_items * 128, rows64 = (uint64_t)n_items * 64;
  if (!make_map3(&mq, qp, p.total_tokens, p.H, 64, false) ||
      !make_map3(&mk, p.k, p.total_tokens, p.H, 64, false) ||
      !make_map3(&mv, p.v, p.total_tokens, p.H, 64, false) ||
      !make_map3(&mg, p.g, p.total_tokens, p.H, 32, true) ||
      !make_map_beta(&mb, p.beta, p.total_tokens, p.H) ||
      !make_map_ws(&mwq, ws.wq, rows128, 128, 128) || !make_map_ws(&mkbt, ws.kbt, rows128, 64, 128) ||
      !make_map_ws(&swq, ws.wq, rows128, 128, 64) || !make_map_ws(&su0, ws.u0, rows64, 128, 64) ||
      !make_map_ws(&so0, ws.o0, rows64, 128, 64, true))
    return set_error(KDA_ERR_CUDA, "tensor-core chunk path: cuTensorMapEncodeTiled failed");
  cudaError_t e =
      cudaFuncSetAttribute(chunk_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, P_SMEM);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(chunk_state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             S_SMEM);
  if (e != cudaSuccess)
    return set_error(KDA_ERR_CUDA, std::string("tensor-core chunk path attribute: ") +
                                       cudaGetErrorString(e));
  const int grid1 = (int)std::min<int64_t>(n_items, sm_count());
  chunk_prep_kernel<<<grid1, kThreads, P_SMEM, s>>>(p, mq, mk, mv, mg, mb, swq, su0, so0, ws,
                                                     (int)n_items);
  count_launches(1);
  kda_status st = check_launch("tensor-core chunk prep kernel");
  if (st != KDA_OK) return st;
  const int cols = p.package ? (p.dk + p.dv) : p.dv;
  dim3 grid2(cols / TW, p.H, p.n_ranges);
  chunk_state_kernel<<<grid2, kThreads, S_SMEM, s>>>(p, mwq, mkbt, ws);
  count_launches(1);
  return check_launch("tensor-core chunk state kernel");
}

}  // namespace kda
