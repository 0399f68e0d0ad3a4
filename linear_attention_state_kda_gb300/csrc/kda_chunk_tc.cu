// Chunked KDA pass on the 5th-generation tensor cores (tcgen05 MMAs, TMEM accumulators,
// TMA-fed shared memory) for bf16 q/k/v with dk = dv = 128.
//
// Chunk algebra (64-token chunk, state S_0 entering it, log-midpoint frame; the same algebra
// as the CUDA-core kernel in kda_chunk_simt.cu, which states it in full):
//   gamma = cumsum(g), rho = gamma_C / 2, Kh = k e^(gamma-rho), Qh = q e^(gamma-rho),
//   Kb = k e^(rho-gamma), Sh = e^rho S_0
//   A    = [Kh; Qh] Kb^T                       (MMA_A: M 128, N 64, K = dk)
//   T    = (I + strict_lower(beta_r A_kk))^-1  (CUDA cores, blocked 16 x 16)
//   W^T  = Kh^T (T diag(beta))^T               (MMA_W: A = Kh^T from TMEM, M = dk, N 64)
//   Ut   = T diag(beta) V                      (MMA_U: N 32, K = 64 tokens)
//   X    = [W; Qh] Sh                          (MMA_X: N 32, K = dk)
//   U    = Ut - X[0:64]
//   O    = X[64:128] + tril(A_qk) U            (MMA_Z accumulates into X)
//   Y    = Kb^T U                              (MMA_Y: A = Kb^T from TMEM, M = dk, N 32)
//   S_C  = e^rho (Sh + Y)                      (since gamma_C - rho = rho)
// Every MMA is kind::tf32 with fp32 accumulation in TMEM, and every shared-memory operand is
// K-major in the 128-byte swizzle (tf32 operands read MN-major came back as zeros on this
// part); the two products that contract over the chunk's tokens with a key-side operand
// on the M side take that operand (Kh^T, Kb^T) from TMEM, where the operand-building threads
// (one per key channel) store it directly. tf32 throughout holds the fp32 state within a few
// 1e-3 of the double-precision recurrence; bf16 operands for the state-touching products
// would not (measured by emulation against the oracle).
//
// A CTA owns one (sequence or segment, head, 32-column tile of the state) and walks the
// range's chunks in order; the tile's 128 x 32 state lives in registers of the first
// warpgroup (thread c holds row c, which is TMEM lane c of the accumulators). q, k and the
// value tile arrive by TMA (two 64-column 128-byte-swizzled boxes each for q and k); g and
// beta are read directly by the per-channel scan. In package mode the CTA runs the same
// chunks on one 32-column tile of the augmented state [M | D] (identity / zero start, zero /
// v values) and produces no outputs.
//
// Waits on mbarriers are bounded (2 s of globaltimer); on expiry the CTA raises
// KDA_STATUS_TIMEOUT, drains its own MMAs and copies (bounded), frees its TMEM and returns.
#include <cuda.h>

#include "kda_internal.cuh"
#include "ptx.cuh"

namespace kda {
namespace {

using namespace ptx;

constexpr int C = kChunk;     // 64 tokens per chunk
constexpr int DK = 128;
constexpr int TW = 32;        // state columns per CTA
constexpr int kThreads = 256;

// shared-memory map (byte offsets from a 1024-byte aligned base)
constexpr uint32_t XA_OFF = 0;                    // [128 rows][128] fp32: [Kh | W ; Qh]
constexpr uint32_t XA_KB = 128 * 128;             //   K-blocks (32 columns) of 16 KiB
constexpr uint32_t KB_OFF = XA_OFF + 4 * XA_KB;   // [64 rows][128] fp32: Kb
constexpr uint32_t KB_KB = 64 * 128;
constexpr uint32_t TQ_OFF = KB_OFF + 4 * KB_KB;   // per K-block: [TB 8K][zeros 8K][Aqk 8K]
constexpr uint32_t TQ_KB = 3 * 8192;
constexpr uint32_t VT_OFF = TQ_OFF + 2 * TQ_KB;   // [32 cols][64 tokens] fp32: V^T
constexpr uint32_t VT_KB = 32 * 128;
constexpr uint32_t UT_OFF = VT_OFF + 2 * VT_KB;   // [32 cols][64 tokens] fp32: U^T
constexpr uint32_t UT_KB = 32 * 128;
constexpr uint32_t SH_OFF = UT_OFF + 2 * UT_KB;   // [32 cols][128] fp32: Sh^T
constexpr uint32_t SH_KB = 32 * 128;
constexpr uint32_t STG_OFF = SH_OFF + 4 * SH_KB;  // TMA staging (also T-solve scratch)
constexpr uint32_t STG_Q = STG_OFF;               // 2 x [64][64] bf16 swizzled boxes
constexpr uint32_t STG_K = STG_OFF + 16384;
constexpr uint32_t STG_V = STG_OFF + 32768;       // [64][32] bf16, unswizzled
constexpr uint32_t STG_BYTES = 36864;
constexpr uint32_t MISC_OFF = STG_OFF + STG_BYTES;
constexpr uint32_t SMEM_BYTES = MISC_OFF + 4096 + 1024;  // + alignment slack

// T-solve scratch inside the staging area (free between the operand build and the next TMA)
constexpr int LA = 65;
constexpr uint32_t SCR_A = STG_OFF;                    // A_kk [64][65] fp32
constexpr uint32_t SCR_X = STG_OFF + 64 * LA * 4;      // X = T [64][65]
constexpr uint32_t SCR_P = STG_OFF + 2 * 64 * LA * 4;  // 3 x [16][16]
static_assert(SCR_P + 3 * 256 * 4 <= STG_OFF + STG_BYTES, "scratch overflow");

// TMEM columns (512 allocated)
constexpr uint32_t TM_A = 0;      // 64: A = [Kh; Qh] Kb^T
constexpr uint32_t TM_WT = 64;    // 64: W^T (lanes = key channels)
constexpr uint32_t TM_U = 128;    // 32: Ut (lanes 0..63 = tokens)
constexpr uint32_t TM_X = 160;    // 32: X, then O in lanes 64..127
constexpr uint32_t TM_Y = 192;    // 32: Y (lanes = key channels)
constexpr uint32_t TM_KHT = 224;  // 64: Kh^T operand (lanes = key channels, columns = tokens)
constexpr uint32_t TM_KBT = 288;  // 64: Kb^T operand

constexpr float kLog2e = 1.4426950408889634f;

struct Misc {
  uint64_t bar_tma, bar_a, bar_w, bar_x, bar_y, bar_drain;
  uint32_t tmem_base;
  int abort;
  float beta[C];
  float part[2][DK];
};

__device__ __forceinline__ void cta_sync() {
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
}

__device__ __forceinline__ float* f32at(uint8_t* base, uint32_t off) {
  return reinterpret_cast<float*>(base + off);
}

__device__ __forceinline__ float bf16at(const uint8_t* base, uint32_t off) {
  return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(base + off));
}

__global__ void __launch_bounds__(kThreads, 1)
chunk_tc_kernel(const __grid_constant__ ChunkParams p, const __grid_constant__ CUtensorMap tmq,
                const __grid_constant__ CUtensorMap tmk,
                const __grid_constant__ CUtensorMap tmv) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  Misc* misc = reinterpret_cast<Misc*>(sm + MISC_OFF);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int qd = warp & 3;                 // TMEM lane quarter of this warp
  const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
  const int tile = blockIdx.x, h = blockIdx.y, sidx = blockIdx.z;
  const int H = p.H;
  const bool pkg = p.package != 0;
  const int j0 = tile * TW;
  const bool mcols = pkg && j0 < DK;
  const int vcol0 = pkg ? j0 - DK : j0;
  const bool has_v = !mcols;
  const int c = tid & (DK - 1), half = tid >> 7;  // operand-building role: channel, token half

  int t_begin = 0, t_end = p.total_tokens;
  if (p.offsets) {
    t_begin = p.offsets[sidx];
    t_end = p.offsets[sidx + 1];
    if (t_end < t_begin || t_begin < 0 || t_end > p.total_tokens) {
      if (tid == 0 && p.status) atomicOr(p.status, KDA_STATUS_BAD_OFFSETS);
      t_end = t_begin;
    }
  }
  const uint32_t tx_bytes = (pkg ? 0u : 16384u) + 16384u + 4096u;

  // ---- one-time setup
  if (warp == 0) {
    tmem_alloc(&misc->tmem_base, 512);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(&misc->bar_tma, 1);
    mbar_init(&misc->bar_a, 1);
    mbar_init(&misc->bar_w, 1);
    mbar_init(&misc->bar_x, 1);
    mbar_init(&misc->bar_y, 1);
    mbar_init(&misc->bar_drain, 1);
    misc->abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmk);
    tma_prefetch_desc(&tmv);
    if (!pkg) tma_prefetch_desc(&tmq);
  }
  // zero block of the TB / Aqk region (rows 64..127 of TB == rows 0..63 of the Aqk view)
  for (uint32_t e = tid; e < 2 * 2048; e += kThreads) {
    const uint32_t kb = e >> 11, w = e & 2047;
    f32at(sm, TQ_OFF + kb * TQ_KB + 8192)[w] = 0.0f;
  }
  if (pkg) {  // no queries: the Qh rows and the A_qk block stay zero
    for (uint32_t e = tid; e < 4 * 2048; e += kThreads) {
      const uint32_t kb = e >> 11, w = e & 2047;
      f32at(sm, XA_OFF + kb * XA_KB + 8192)[w] = 0.0f;
    }
    for (uint32_t e = tid; e < 2 * 2048; e += kThreads) {
      const uint32_t kb = e >> 11, w = e & 2047;
      f32at(sm, TQ_OFF + kb * TQ_KB + 16384)[w] = 0.0f;
    }
  }
  // state tile: thread c < 128 holds row c
  float S[TW], Sh[TW], Ut[TW];
#pragma unroll
  for (int j = 0; j < TW; ++j) {
    float x = 0.0f;
    if (tid < DK) {
      if (pkg) x = (mcols && tid == j0 + j) ? 1.0f : 0.0f;
      else if (p.init) x = p.init[(((int64_t)sidx * H + h) * DK + tid) * DK + j0 + j];
    }
    S[j] = x;
    Sh[j] = 0.0f;
    Ut[j] = 0.0f;
  }
  cta_sync();
  const uint32_t tbase = misc->tmem_base;
  const uint32_t sbase = smem_u32(sm);

  auto issue_tma = [&](int t0) {
    mbar_arrive_expect_tx(&misc->bar_tma, tx_bytes);
    if (!pkg) {
      tma_load_3d(sm + STG_Q, &tmq, &misc->bar_tma, 0, h, t0);
      tma_load_3d(sm + STG_Q + 8192, &tmq, &misc->bar_tma, 64, h, t0);
    }
    tma_load_3d(sm + STG_K, &tmk, &misc->bar_tma, 0, h, t0);
    tma_load_3d(sm + STG_K + 8192, &tmk, &misc->bar_tma, 64, h, t0);
    tma_load_3d(sm + STG_V, &tmv, &misc->bar_tma, vcol0 < 0 ? 0 : vcol0, h, t0);
  };
  bool tma_out = false;  // thread 0: a load is in flight, completing phase parity tma_par
  uint32_t tma_par = 0;
  if (tid == 0 && t_end > t_begin) {
    issue_tma(t_begin);
    tma_out = true;
  }

  uint32_t it = 0;
  bool ok = true;
  for (int t0 = t_begin; t0 < t_end; t0 += C, ++it) {
    const int n = min(C, t_end - t0);
    const uint32_t par = it & 1u;
    // ================= Ph1: decay, operands, state in the midpoint frame
    float gl[32];
    float acc = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const int r = half * 32 + i;
      gl[i] = (r < n) ? p.g[((int64_t)(t0 + r) * H + h) * DK + c] * kLog2e : 0.0f;
      acc += gl[i];
    }
    misc->part[half][c] = acc;
    if (tid < C) misc->beta[tid] = (tid < n) ? p.beta[(int64_t)(t0 + tid) * H + h] : 0.0f;
    __syncthreads();
    const float p0 = misc->part[0][c], p1 = misc->part[1][c];
    const float rho2 = 0.5f * (p0 + p1);  // log2 units
    if (half == 0 && !((p0 + p1) >= -kMaxChunkDecay * kLog2e) && p.status)
      atomicOr(p.status, KDA_STATUS_DECAY_RANGE);
    if (!mbar_wait(&misc->bar_tma, par)) misc->abort = 1;
    else tma_out = false;
    __syncthreads();
    if (misc->abort) { ok = false; break; }
    {
      float gam = half ? p0 : 0.0f;
#pragma unroll
      for (int blk = 0; blk < 2; ++blk) {
        float kh[16], kb[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int r = half * 32 + blk * 16 + i;
          gam += gl[blk * 16 + i];
          const float x = gam - rho2;
          const float e1 = exp2f(x), e2 = exp2f(-x);
          float kv = 0.0f, qv = 0.0f;
          if (r < n) {
            kv = bf16at(sm, STG_K + sw128_off16(r, c, 8192));
            if (!pkg) qv = bf16at(sm, STG_Q + sw128_off16(r, c, 8192));
          }
          kh[i] = kv * e1;
          kb[i] = kv * e2;
          *f32at(sm, XA_OFF + sw128_off32(r, c, XA_KB)) = kh[i];
          if (!pkg) *f32at(sm, XA_OFF + sw128_off32(64 + r, c, XA_KB)) = qv * e1;
          *f32at(sm, KB_OFF + sw128_off32(r, c, KB_KB)) = kb[i];
        }
        // Kh^T and Kb^T as TMEM operands: lane = channel c, column = token
        tmem_st16(tbase + lane_base + TM_KHT + half * 32 + blk * 16, kh);
        tmem_st16(tbase + lane_base + TM_KBT + half * 32 + blk * 16, kb);
      }
      tmem_st_wait();
    }
    for (int e = tid; e < C * TW; e += kThreads) {  // V^T: row = value column, K = token
      const int j = e >> 6, r = e & 63;
      float x = 0.0f;
      if (r < n && has_v) x = bf16at(sm, STG_V + r * 64 + j * 2);
      *f32at(sm, VT_OFF + sw128_off32(j, r, VT_KB)) = x;
    }
    float erho = 1.0f;
    if (tid < DK) {
      erho = exp2f(rho2);
#pragma unroll
      for (int j = 0; j < TW; ++j) {
        Sh[j] = erho * S[j];
        *f32at(sm, SH_OFF + sw128_off32(j, c, SH_KB)) = Sh[j];
      }
    }
    fence_proxy_async_smem();
    cta_sync();
    // ================= Ph2: A = [Kh; Qh] Kb^T
    if (tid == 0) {
      const uint32_t idesc = idesc_make(kFmtTF32, 128, 64, false, false);
#pragma unroll
      for (int s = 0; s < 16; ++s) {
        const uint64_t a = sdesc_sw128(sbase + XA_OFF + (s >> 2) * XA_KB + (s & 3) * 32, 16, 1024);
        const uint64_t b = sdesc_sw128(sbase + KB_OFF + (s >> 2) * KB_KB + (s & 3) * 32, 16, 1024);
        mma_tf32(tbase + TM_A, a, b, idesc, s > 0);
      }
      mma_commit(&misc->bar_a);
    }
    if (!mbar_wait(&misc->bar_a, par)) misc->abort = 1;
    tc_fence_after();
    // ================= Ph3: A_kk -> scratch, A_qk -> operand, then T
    {
      float v[32];
      const int ch = warp >> 2;
      tmem_ld32(tbase + lane_base + TM_A + ch * 32, v);
      const int R = qd * 32 + lane;
      if (R < C) {
        const float br = misc->beta[R];
        float* Akk = f32at(sm, SCR_A);
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int i = ch * 32 + j;
          Akk[R * LA + i] = (i < R) ? br * v[j] : 0.0f;
        }
      } else if (!pkg) {
        const int r = R - C;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int i = ch * 32 + j;
          *f32at(sm, TQ_OFF + 8192 + sw128_off32(C + r, i, TQ_KB)) = (i <= r) ? v[j] : 0.0f;
        }
      }
    }
    cta_sync();
    if (misc->abort) { ok = false; break; }
    {
      float* Akk = f32at(sm, SCR_A);
      float* X = f32at(sm, SCR_X);
      float* P = f32at(sm, SCR_P);
      // diagonal 16 x 16 blocks: lane i of a 16-lane group owns column i of its block
      if (tid < 64) {
        const int blk = tid >> 4, i = tid & 15, I0 = blk * 16;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
          float a = 0.0f;
#pragma unroll
          for (int l = 0; l < r; ++l) a = fmaf(Akk[(I0 + r) * LA + I0 + l], x[l], a);
          x[r] = (r < i) ? 0.0f : (r == i ? 1.0f : -a);
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) X[(I0 + r) * LA + I0 + i] = x[r];
      }
      // blocks above the diagonal are zero
      for (int e = tid; e < 64 * 64; e += kThreads) {
        const int r = e >> 6, i = e & 63;
        if ((i >> 4) > (r >> 4)) X[r * LA + i] = 0.0f;
      }
      __syncthreads();
      // off-diagonal blocks by distance: X_IJ = -X_II * sum_{L=J}^{I-1} A_IL X_LJ
      for (int dist = 1; dist < 4; ++dist) {
        const int nb = 4 - dist;
        for (int e = tid; e < nb * 256; e += kThreads) {
          const int b = e >> 8, rr = (e >> 4) & 15, cc = e & 15;
          const int J = b, I = b + dist;
          float a = 0.0f;
          for (int L = J; L < I; ++L)
#pragma unroll
            for (int l = 0; l < 16; ++l)
              a = fmaf(Akk[(I * 16 + rr) * LA + L * 16 + l], X[(L * 16 + l) * LA + J * 16 + cc],
                       a);
          P[b * 256 + rr * 16 + cc] = a;
        }
        __syncthreads();
        for (int e = tid; e < nb * 256; e += kThreads) {
          const int b = e >> 8, rr = (e >> 4) & 15, cc = e & 15;
          const int J = b, I = b + dist;
          float a = 0.0f;
#pragma unroll
          for (int l = 0; l < 16; ++l)
            a = fmaf(X[(I * 16 + rr) * LA + I * 16 + l], P[b * 256 + l * 16 + cc], a);
          X[(I * 16 + rr) * LA + J * 16 + cc] = -a;
        }
        __syncthreads();
      }
      // T diag(beta) into the TB operand (K-major: row = token r, K = token i)
      for (int e = tid; e < C * C; e += kThreads) {
        const int r = e >> 6, i = e & 63;
        const float x = (i <= r) ? X[r * LA + i] * misc->beta[i] : 0.0f;
        *f32at(sm, TQ_OFF + sw128_off32(r, i, TQ_KB)) = x;
      }
    }
    fence_proxy_async_smem();
    cta_sync();
    // ================= Ph4: W^T = Kh^T TB^T, Ut = TB V; then prefetch the next chunk
    if (tid == 0) {
      const uint32_t idw = idesc_make(kFmtTF32, 128, 64, false, false);
      const uint32_t idu = idesc_make(kFmtTF32, 128, 32, false, false);
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        const uint64_t tb = sdesc_sw128(sbase + TQ_OFF + (s >> 2) * TQ_KB + (s & 3) * 32, 16, 1024);
        mma_tf32_ts(tbase + TM_WT, tbase + TM_KHT + s * 8, tb, idw, s > 0);
        if (has_v) {
          const uint64_t bv = sdesc_sw128(sbase + VT_OFF + (s >> 2) * VT_KB + (s & 3) * 32, 16, 1024);
          mma_tf32(tbase + TM_U, tb, bv, idu, s > 0);
        }
      }
      mma_commit(&misc->bar_w);
      if (t0 + C < t_end) {
        issue_tma(t0 + C);
        tma_out = true;
        tma_par = (it + 1) & 1u;
      }
    }
    if (!mbar_wait(&misc->bar_w, par)) misc->abort = 1;
    tc_fence_after();
    // ================= Ph5: W into the Kh rows of XA; Ut into registers
    {
      float v[32];
      const int ch = warp >> 2;  // token half
      tmem_ld32(tbase + lane_base + TM_WT + ch * 32, v);
#pragma unroll
      for (int j = 0; j < 32; ++j)
        *f32at(sm, XA_OFF + sw128_off32(ch * 32 + j, c, XA_KB)) = v[j];
      if (warp < 2 && has_v) tmem_ld32(tbase + lane_base + TM_U, Ut);
    }
    fence_proxy_async_smem();
    cta_sync();
    if (misc->abort) { ok = false; break; }
    // ================= Ph6: X = [W; Qh] Sh
    if (tid == 0) {
      const uint32_t idx = idesc_make(kFmtTF32, 128, 32, false, false);
#pragma unroll
      for (int s = 0; s < 16; ++s) {
        const uint64_t a = sdesc_sw128(sbase + XA_OFF + (s >> 2) * XA_KB + (s & 3) * 32, 16, 1024);
        const uint64_t b = sdesc_sw128(sbase + SH_OFF + (s >> 2) * SH_KB + (s & 3) * 32, 16, 1024);
        mma_tf32(tbase + TM_X, a, b, idx, s > 0);
      }
      mma_commit(&misc->bar_x);
    }
    if (!mbar_wait(&misc->bar_x, par)) misc->abort = 1;
    tc_fence_after();
    if (warp < 2) {  // token rows 0..63: U = Ut - W Sh, stored as U^T (K-major)
      float x[32];
      tmem_ld32(tbase + lane_base + TM_X, x);
      const int r = qd * 32 + lane;
#pragma unroll
      for (int j = 0; j < TW; ++j) *f32at(sm, UT_OFF + sw128_off32(j, r, UT_KB)) = Ut[j] - x[j];
    }
    fence_proxy_async_smem();
    cta_sync();
    if (misc->abort) { ok = false; break; }
    // ================= Ph7: Y = Kb^T U, O = X_q + tril(A_qk) U
    if (tid == 0) {
      const uint32_t idy = idesc_make(kFmtTF32, 128, 32, false, false);
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        const uint64_t b = sdesc_sw128(sbase + UT_OFF + (s >> 2) * UT_KB + (s & 3) * 32, 16, 1024);
        mma_tf32_ts(tbase + TM_Y, tbase + TM_KBT + s * 8, b, idy, s > 0);
        if (!pkg) {
          const uint64_t az =
              sdesc_sw128(sbase + TQ_OFF + 8192 + (s >> 2) * TQ_KB + (s & 3) * 32, 16, 1024);
          mma_tf32(tbase + TM_X, az, b, idy, 1);
        }
      }
      mma_commit(&misc->bar_y);
    }
    if (!mbar_wait(&misc->bar_y, par)) misc->abort = 1;
    tc_fence_after();
    if (warp >= 2 && warp < 4 && !pkg && p.o) {  // output rows (Qh rows 64..127)
      float x[32];
      tmem_ld32(tbase + lane_base + TM_X, x);
      const int r = qd * 32 + lane - C;
      if (r < n) {
        __nv_bfloat16* o = (__nv_bfloat16*)p.o + ((int64_t)(t0 + r) * H + h) * DK + j0;
#pragma unroll
        for (int j = 0; j < TW; j += 8) {
          uint4 pk;
          __nv_bfloat162 b0 = __floats2bfloat162_rn(p.scale * x[j], p.scale * x[j + 1]);
          __nv_bfloat162 b1 = __floats2bfloat162_rn(p.scale * x[j + 2], p.scale * x[j + 3]);
          __nv_bfloat162 b2 = __floats2bfloat162_rn(p.scale * x[j + 4], p.scale * x[j + 5]);
          __nv_bfloat162 b3 = __floats2bfloat162_rn(p.scale * x[j + 6], p.scale * x[j + 7]);
          pk.x = *reinterpret_cast<uint32_t*>(&b0);
          pk.y = *reinterpret_cast<uint32_t*>(&b1);
          pk.z = *reinterpret_cast<uint32_t*>(&b2);
          pk.w = *reinterpret_cast<uint32_t*>(&b3);
          *reinterpret_cast<uint4*>(o + j) = pk;
        }
      }
    }
    if (tid < DK) {  // state rows: S = e^rho (Sh + Y)
      float y[32];
      tmem_ld32(tbase + lane_base + TM_Y, y);
#pragma unroll
      for (int j = 0; j < TW; ++j) S[j] = erho * (Sh[j] + y[j]);
    }
    cta_sync();
    if (misc->abort) { ok = false; break; }
  }
  // ---- exit state of this tile
  if (!ok) {
    // Let this CTA's in-flight MMAs and prefetch drain (bounded) before its shared memory
    // and TMEM are released.
    if (tid == 0) {
      if (p.status) atomicOr(p.status, KDA_STATUS_TIMEOUT);
      mma_commit(&misc->bar_drain);
      mbar_wait(&misc->bar_drain, 0, 100000000ull);
      if (tma_out) mbar_wait(&misc->bar_tma, tma_par, 100000000ull);
    }
  } else if (tid < DK) {
    const int64_t sh = (int64_t)sidx * H + h;
#pragma unroll
    for (int j = 0; j < TW; ++j) {
      if (pkg) {
        if (mcols) p.M[(sh * DK + tid) * DK + j0 + j] = S[j];
        else p.D[(sh * DK + tid) * DK + vcol0 + j] = S[j];
      } else if (p.final_state) {
        p.final_state[(sh * DK + tid) * DK + j0 + j] = S[j];
      }
    }
  }
  cta_sync();
  if (warp == 0) tmem_dealloc(tbase, 512);
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

// [T, H, d] bf16 viewed as a 3-D tensor (d, H, T); box (box_d, 1, 64 tokens).
bool make_map(CUtensorMap* m, const void* ptr, int T, int H, int d, int box_d, bool swizzle) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)(T > 0 ? T : 1)};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)H * d * 2};
  cuuint32_t box[3] = {(cuuint32_t)box_d, 1, (cuuint32_t)C};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides,
                   box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace

bool chunk_tc_supported(const ChunkParams& p, kda_dtype dt) {
  return dt == KDA_BF16 && p.dk == 128 && p.dv == 128 && p.total_tokens > 0 &&
         encode_fn() != nullptr;
}

kda_status launch_chunk_tc(const ChunkParams& p, kda_dtype dt, cudaStream_t s) {
  (void)dt;
  if (p.n_ranges == 0) return KDA_OK;
  CUtensorMap mq, mk, mv;
  const void* qp = p.q ? p.q : p.k;
  if (!make_map(&mq, qp, p.total_tokens, p.H, 128, 64, true) ||
      !make_map(&mk, p.k, p.total_tokens, p.H, 128, 64, true) ||
      !make_map(&mv, p.v, p.total_tokens, p.H, 128, TW, false))
    return set_error(KDA_ERR_CUDA, "tensor-core chunk kernel: cuTensorMapEncodeTiled failed");
  cudaError_t e = cudaFuncSetAttribute(chunk_tc_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess)
    return set_error(KDA_ERR_CUDA, std::string("tensor-core chunk kernel attribute: ") +
                                       cudaGetErrorString(e));
  const int cols = p.package ? (p.dk + p.dv) : p.dv;
  dim3 grid(cols / TW, p.H, p.n_ranges);
  chunk_tc_kernel<<<grid, kThreads, SMEM_BYTES, s>>>(p, mq, mk, mv);
  count_launches(1);
  return check_launch("tensor-core chunk kernel");
}

}  // namespace kda
