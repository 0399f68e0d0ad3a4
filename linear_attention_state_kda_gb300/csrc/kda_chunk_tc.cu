// Chunked KDA pass on the 5th-generation tensor cores (tcgen05 MMAs, TMEM accumulators,
// TMA-fed shared memory) for bf16 q/k/v with dk = dv = 128.
//
// Chunk algebra (64-token chunk, state S_0 entering it, log-midpoint frame; the same algebra
// as the CUDA-core kernel in kda_chunk_simt.cu, which states it in full):
//   gamma = cumsum(g), rho = gamma_C / 2, Kh = k e^(gamma-rho), Qh = q e^(gamma-rho),
//   Kb = k e^(rho-gamma), Sh = e^rho S_0, T = (I + strict_lower(beta_r Kh Kb^T))^-1
//   U   = T diag(beta) V - T diag(beta) Kh Sh = TB (V - Kh Sh)           (TB = T diag(beta))
//   O   = Qh Sh + tril(Qh Kb^T) U,    S_C = e^rho (Sh + Kb^T U)
// Forming V - Kh Sh in fp32 before the product with TB (instead of subtracting two separately
// rounded products TB V and (TB Kh) Sh) both removes a product and avoids cancellation.
// Per chunk, three tensor-core rounds (all kind::tf32, fp32 accumulation in TMEM):
//   round 1: A = [Kh; Qh] Kb^T (M 128, N 64, K = dk) and X = [Kh; Qh] Sh (M 128, N 32)
//   round 2: U = TB (V - X[0:64])                  (A = TB from TMEM, K = 64 tokens)
//   round 3: Y = Kb^T U  (A = Kb^T from TMEM)  and  X[64:128] += tril(A_qk) U  (A from TMEM)
// with the T solve (CUDA cores, blocked 16 x 16) between rounds 1 and 2. Every shared-memory
// operand is K-major in the 128-byte swizzle (tf32 operands read MN-major came back as zeros
// on this part); operands needed in the other orientation are staged in TMEM by the threads
// that produce them. tf32 throughout holds the fp32 state within a few 1e-3 of the
// double-precision recurrence; bf16 operands for the state-touching products would not
// (measured by emulation against the oracle).
//
// A CTA owns one (sequence or segment, head, 32-column tile of the state) and walks the
// range's chunks in order. The tile's 128 x 32 state lives in TMEM (lane = key channel).
// q, k, v, g and beta of a chunk arrive by TMA (q and k as two 64-column 128-byte-swizzled
// boxes each); the next chunk's loads are issued as soon as the staging buffer is free. In
// package mode the CTA runs the same chunks on one 32-column tile of the augmented state
// [M | D] (identity / zero start, zero / v values) and produces no outputs.
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
constexpr uint32_t XA_OFF = 0;                    // [128 rows][128] fp32: [Kh ; Qh]
constexpr uint32_t XA_KB = 128 * 128;             //   K-blocks (32 columns) of 16 KiB
constexpr uint32_t KB_OFF = XA_OFF + 4 * XA_KB;   // [64 rows][128] fp32: Kb
constexpr uint32_t KB_KB = 64 * 128;
constexpr uint32_t VT_OFF = KB_OFF + 4 * KB_KB;   // [32 cols][64 tokens] fp32: (V - Kh Sh)^T
constexpr uint32_t VT_KB = 32 * 128;
constexpr uint32_t UT_OFF = VT_OFF + 2 * VT_KB;   // [32 cols][64 tokens] fp32: U^T
constexpr uint32_t UT_KB = 32 * 128;
constexpr uint32_t SH_OFF = UT_OFF + 2 * UT_KB;   // [32 cols][128] fp32: Sh^T
constexpr uint32_t SH_KB = 32 * 128;
constexpr uint32_t STG_OFF = SH_OFF + 4 * SH_KB;  // TMA staging (also T-solve scratch)
constexpr uint32_t STG_Q = STG_OFF;               // 2 x [64][64] bf16 swizzled boxes
constexpr uint32_t STG_K = STG_OFF + 16384;
constexpr uint32_t STG_V = STG_OFF + 32768;       // [64][32] bf16
constexpr uint32_t STG_G = STG_OFF + 36864;       // [64][128] fp32
constexpr uint32_t STG_B = STG_OFF + 69632;       // [64][4] fp32 (beta of 4 heads)
constexpr uint32_t STG_BYTES = 70656;
constexpr uint32_t MISC_OFF = STG_OFF + STG_BYTES;
constexpr uint32_t SMEM_BYTES = MISC_OFF + 2048 + 1024;  // + alignment slack

// T-solve scratch inside the staging area (q, k, v and g are consumed by then; the next
// chunk's loads are issued after the solve). Rows padded to 68 floats: 16-byte aligned rows
// whose banks shift by 4 per row. SCR_A does not overlap the value staging, SCR_X does.
constexpr int LA = 68;
constexpr uint32_t SCR_A = STG_OFF;                    // beta_r A_kk [64][68] fp32
constexpr uint32_t SCR_X = STG_OFF + 64 * LA * 4;      // X = (I + A_kk)^-1 [64][68]
constexpr uint32_t SCR_P = STG_OFF + 2 * 64 * LA * 4;  // 3 x [16][16] partial products
static_assert(SCR_P + 3 * 256 * 4 <= STG_B, "scratch overflow");
static_assert(SCR_A + 64 * LA * 4 <= STG_V, "A_kk scratch must not overlap the value tile");

// TMEM columns (512 allocated)
// (A and Kb^T are double-buffered: the next chunk's are built while round 3 reads these.)
constexpr uint32_t TM_A0 = 0;     // 2 x 64: [Kh; Qh] Kb^T; lanes 64..127 masked to tril(A_qk)
constexpr uint32_t TM_X = 128;    // 32: [Kh; Qh] Sh, then O in lanes 64..127
constexpr uint32_t TM_U = 160;    // 32: U (lanes 0..63 = tokens)
constexpr uint32_t TM_Y = 192;    // 32: Kb^T U (lanes = key channels)
constexpr uint32_t TM_KBT0 = 224; // 2 x 64: Kb^T operand (lanes = key channels, cols = tokens)
constexpr uint32_t TM_TB = 352;   // 64: TB operand (lanes 0..63 = tokens; 64..127 zero)
constexpr uint32_t TM_S = 416;    // 32: state tile (lanes = key channels)

constexpr float kLog2e = 1.4426950408889634f;

struct Misc {
  uint64_t bar_tma, bar_a, bar_x, bar_2, bar_3, bar_drain;
  uint32_t tmem_base;
  int abort;
  float part[2][DK];
  float beta[C];
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
                const __grid_constant__ CUtensorMap tmv,
                const __grid_constant__ CUtensorMap tmg,
                const __grid_constant__ CUtensorMap tmb) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  Misc* misc = reinterpret_cast<Misc*>(sm + MISC_OFF);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int qd = warp & 3;                 // TMEM lane quarter of this warp
  const int ch = warp >> 2;                // column half of this warp in TMEM reads
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
  const uint32_t tx_bytes = (pkg ? 0u : 16384u) + 16384u + 4096u + 32768u + 1024u;

  // ---- one-time setup
  if (warp == 0) {
    tmem_alloc(&misc->tmem_base, 512);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(&misc->bar_tma, 1);
    mbar_init(&misc->bar_a, 1);
    mbar_init(&misc->bar_x, 1);
    mbar_init(&misc->bar_2, 1);
    mbar_init(&misc->bar_3, 1);
    mbar_init(&misc->bar_drain, 1);
    misc->abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmk);
    tma_prefetch_desc(&tmv);
    tma_prefetch_desc(&tmg);
    tma_prefetch_desc(&tmb);
    if (!pkg) tma_prefetch_desc(&tmq);
  }
  if (pkg) {  // no queries: the Qh rows stay zero
    for (uint32_t e = tid; e < 4 * 2048; e += kThreads) {
      const uint32_t kb = e >> 11, w = e & 2047;
      f32at(sm, XA_OFF + kb * XA_KB + 8192)[w] = 0.0f;
    }
  }
  cta_sync();
  const uint32_t tbase = misc->tmem_base;
  const uint32_t sbase = smem_u32(sm);
  {
    // state tile into TMEM (lane = row c; warps 0-3 columns 0..15, warps 4-7 16..31), and
    // zeros into the padding lanes 64..127 of the TB operand
    float v[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int col = ch * 16 + j;
      float x = 0.0f;
      if (pkg) x = (mcols && c == j0 + col) ? 1.0f : 0.0f;
      else if (p.init) x = p.init[(((int64_t)sidx * H + h) * DK + c) * DK + j0 + col];
      v[j] = x;
    }
    tmem_st16(tbase + lane_base + TM_S + ch * 16, v);
    if (qd >= 2) {
#pragma unroll
      for (int j = 0; j < 16; ++j) v[j] = 0.0f;
      tmem_st16(tbase + lane_base + TM_TB + ch * 32, v);
      tmem_st16(tbase + lane_base + TM_TB + ch * 32 + 16, v);
    }
    tmem_st_wait();
  }

  auto issue_tma = [&](int t0) {
    mbar_arrive_expect_tx(&misc->bar_tma, tx_bytes);
    if (!pkg) {
      tma_load_3d(sm + STG_Q, &tmq, &misc->bar_tma, 0, h, t0);
      tma_load_3d(sm + STG_Q + 8192, &tmq, &misc->bar_tma, 64, h, t0);
    }
    tma_load_3d(sm + STG_K, &tmk, &misc->bar_tma, 0, h, t0);
    tma_load_3d(sm + STG_K + 8192, &tmk, &misc->bar_tma, 64, h, t0);
    tma_load_3d(sm + STG_V, &tmv, &misc->bar_tma, vcol0 < 0 ? 0 : vcol0, h, t0);
    tma_load_3d(sm + STG_G, &tmg, &misc->bar_tma, 0, h, t0);
    tma_load_2d(sm + STG_B, &tmb, &misc->bar_tma, h & ~3, t0);
  };
  bool tma_out = false;  // thread 0: a load is in flight, completing phase parity tma_par
  uint32_t tma_par = 0;
  if (tid == 0 && t_end > t_begin) {
    issue_tma(t_begin);
    tma_out = true;
  }
  cta_sync();

  const float* gs = f32at(sm, STG_G);
  const float* bs4 = f32at(sm, STG_B);
  const int hb = h & 3;

  // Operand build of one chunk (state-independent): waits for its loads, forms the decay
  // prefix, writes Kh, Qh (XA), Kb (KB) and Kb^T (TMEM buffer kbuf); returns this thread's
  // channel's rho in log2 units. Whole-CTA; sets misc->abort on a timed-out load.
  auto build = [&](int tc0, uint32_t itc) -> float {
    const int n = min(C, t_end - tc0);
    const uint32_t kbt = TM_KBT0 + (itc & 1u) * 64u;
    if (!mbar_wait(&misc->bar_tma, itc & 1u)) misc->abort = 1;
    else tma_out = false;
    const int nv = n - half * 32;  // valid rows in this thread's half
    float gl[32];
    float acc = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      gl[i] = (i < nv) ? gs[(half * 32 + i) * DK + c] * kLog2e : 0.0f;
      acc += gl[i];
    }
    misc->part[half][c] = acc;
    if (tid < C) misc->beta[tid] = (tid < n) ? bs4[tid * 4 + hb] : 0.0f;
    __syncthreads();
    const float p0 = misc->part[0][c], p1 = misc->part[1][c];
    const float rho2 = 0.5f * (p0 + p1);  // log2 units
    if (half == 0 && !((p0 + p1) >= -kMaxChunkDecay * kLog2e) && p.status)
      atomicOr(p.status, KDA_STATUS_DECAY_RANGE);
    {
      // Row r = 32 half + t of every tile below: (r >> 3) and (r & 7) are compile-time per t,
      // so each swizzled address is a per-thread base plus a constant and one XOR.
      const uint32_t b16 = STG_K + (c >> 6) * 8192 + (c & 7) * 2 + half * 4096;
      const uint32_t x16 = (c & 63) >> 3;
      const uint32_t bxa = XA_OFF + (c >> 5) * XA_KB + (c & 3) * 4 + half * 4096;
      const uint32_t bkb = KB_OFF + (c >> 5) * KB_KB + (c & 3) * 4 + half * 4096;
      const uint32_t x32 = (c & 31) >> 2;
      float gam = half ? p0 : 0.0f;
#pragma unroll
      for (int blk = 0; blk < 2; ++blk) {
        float kb[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int t = blk * 16 + i;
          const uint32_t row = (uint32_t)(t >> 3) * 1024u + (uint32_t)(t & 7) * 128u;
          gam += gl[t];
          const float x = gam - rho2;
          const float e1 = ex2_approx(x), e2 = ex2_approx(-x);
          float kv = 0.0f, qv = 0.0f;
          if (t < nv) {
            const uint32_t o16 = b16 + row + ((x16 ^ (uint32_t)(t & 7)) << 4);
            kv = bf16at(sm, o16);
            if (!pkg) qv = bf16at(sm, o16 - (STG_K - STG_Q));
          }
          kb[i] = kv * e2;
          const uint32_t sw = row + ((x32 ^ (uint32_t)(t & 7)) << 4);
          *f32at(sm, bxa + sw) = kv * e1;
          if (!pkg) *f32at(sm, bxa + 8192 + sw) = qv * e1;
          *f32at(sm, bkb + sw) = kb[i];
        }
        // Kb^T as the TMEM operand of round 3: lane = channel c, column = token
        tmem_st16(tbase + lane_base + kbt + half * 32 + blk * 16, kb);
      }
    }
    tmem_st_wait();
    return rho2;
  };
  // A = [Kh; Qh] Kb^T of a built chunk into TMEM buffer (itc & 1); thread 0.
  auto issue_a = [&](uint32_t itc) {
    const uint32_t ida = idesc_make(kFmtTF32, 128, 64, false, false);
#pragma unroll
    for (int s = 0; s < 16; ++s) {
      const uint64_t a = sdesc_sw128(sbase + XA_OFF + (s >> 2) * XA_KB + (s & 3) * 32, 16, 1024);
      const uint64_t b = sdesc_sw128(sbase + KB_OFF + (s >> 2) * KB_KB + (s & 3) * 32, 16, 1024);
      mma_tf32(tbase + TM_A0 + (itc & 1u) * 64u, a, b, ida, s > 0);
    }
    mma_commit(&misc->bar_a);
  };

  uint32_t it = 0;
  bool ok = true;
  float rho2 = 0.0f;
  if (t_end > t_begin) {
    rho2 = build(t_begin, 0);
    fence_proxy_async_smem();
    cta_sync();
    if (misc->abort) ok = false;
    else if (tid == 0) issue_a(0);
  }
  for (int t0 = t_begin; ok && t0 < t_end; t0 += C, ++it) {
    const int n = min(C, t_end - t0);
    const uint32_t par = it & 1u;
    const uint32_t tma_a = TM_A0 + par * 64u, tm_kbt = TM_KBT0 + par * 64u;
    // ================= Ph1: state in the midpoint frame (operands were built earlier)
    const float erho = ex2_approx(rho2);
    {  // Sh = e^rho S into the round-1 operand (lane c; warps 0-3 cols 0..15, 4-7 16..31)
      float s[16];
      tmem_ld16(tbase + lane_base + TM_S + ch * 16, s);
      const uint32_t bsh = SH_OFF + (c >> 5) * SH_KB + (c & 3) * 4 + (uint32_t)ch * 2048;
      const uint32_t xs = (c & 31) >> 2;
#pragma unroll
      for (int j = 0; j < 16; ++j)
        *f32at(sm, bsh + (uint32_t)(j >> 3) * 1024u + (uint32_t)(j & 7) * 128u +
                       ((xs ^ (uint32_t)(j & 7)) << 4)) = erho * s[j];
    }
    fence_proxy_async_smem();
    cta_sync();
    // ================= round 1: X = [Kh; Qh] Sh (A of this chunk is already in flight)
    if (tid == 0) {
      const uint32_t idx = idesc_make(kFmtTF32, 128, 32, false, false);
#pragma unroll
      for (int s = 0; s < 16; ++s) {
        const uint64_t a = sdesc_sw128(sbase + XA_OFF + (s >> 2) * XA_KB + (s & 3) * 32, 16, 1024);
        const uint64_t bs = sdesc_sw128(sbase + SH_OFF + (s >> 2) * SH_KB + (s & 3) * 32, 16, 1024);
        mma_tf32(tbase + TM_X, a, bs, idx, s > 0);
      }
      mma_commit(&misc->bar_x);
    }
    if (!mbar_wait(&misc->bar_a, par)) misc->abort = 1;
    tc_fence_after();
    // ================= Ph3: A_kk -> scratch, A_qk masked in place, V - Kh Sh -> operand
    {
      float v[32];
      tmem_ld32(tbase + lane_base + tma_a + ch * 32, v);
      const int R = qd * 32 + lane;
      if (R < C) {  // beta_r A_kk, strictly lower, as 16-byte row segments
        const float br = misc->beta[R];
        float* arow = f32at(sm, SCR_A) + R * LA + ch * 32;
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
          const int i = ch * 32 + j;
          *reinterpret_cast<float4*>(arow + j) =
              make_float4(i < R ? br * v[j] : 0.0f, i + 1 < R ? br * v[j + 1] : 0.0f,
                          i + 2 < R ? br * v[j + 2] : 0.0f, i + 3 < R ? br * v[j + 3] : 0.0f);
        }
      } else {  // causal A_qk (diagonal included), the round-3 operand, rewritten in TMEM
        const int r = R - C;
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = (ch * 32 + j <= r) ? v[j] : 0.0f;
        tmem_st16(tbase + lane_base + tma_a + ch * 32, v);
        tmem_st16(tbase + lane_base + tma_a + ch * 32 + 16, v + 16);
        tmem_st_wait();
      }
    }
    if (!mbar_wait(&misc->bar_x, par)) misc->abort = 1;
    tc_fence_after();
    if (qd < 2) {
      // (V - Kh Sh) for token R, 16 value columns per warp, stored transposed (K = token)
      const int R = qd * 32 + lane;
      float x[16];
      tmem_ld16(tbase + lane_base + TM_X + ch * 16, x);
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int col = ch * 16 + j;
        const float vv = (R < n && has_v) ? bf16at(sm, STG_V + R * 64 + col * 2) : 0.0f;
        *f32at(sm, VT_OFF + sw128_off32(col, R, VT_KB)) = vv - x[j];
      }
    }
    cta_sync();
    if (misc->abort) { ok = false; break; }
    {
      // T = (I + A_kk)^-1 in 16 x 16 blocks
      const float* Akk = f32at(sm, SCR_A);
      float* X = f32at(sm, SCR_X);
      float* P = f32at(sm, SCR_P);
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
        // blocks above the diagonal are zero (read by the TB copy below)
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
      // product P passing through a per-warp 16 x 8 tile of shared memory.
      {
        const int gq = lane >> 2, tq = lane & 3;
        float* Pw = P + warp * 128;  // [16][8]
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
      // TB = T diag(beta) into TMEM lanes 0..63 (the round-2 A operand)
      if (qd < 2) {
        const int r = qd * 32 + lane;
        const float* xrow = X + r * LA + ch * 32;
        const float* bt = misc->beta + ch * 32;
        float v[32];
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
          const float4 t4 = *reinterpret_cast<const float4*>(xrow + j);
          v[j] = t4.x * bt[j];
          v[j + 1] = t4.y * bt[j + 1];
          v[j + 2] = t4.z * bt[j + 2];
          v[j + 3] = t4.w * bt[j + 3];
        }
        tmem_st16(tbase + lane_base + TM_TB + ch * 32, v);
        tmem_st16(tbase + lane_base + TM_TB + ch * 32 + 16, v + 16);
        tmem_st_wait();
      }
    }
    fence_proxy_async_smem();
    cta_sync();
    // ================= round 2: U = TB (V - Kh Sh); then load the next chunk
    if (tid == 0) {
      const uint32_t idu = idesc_make(kFmtTF32, 128, 32, false, false);
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        const uint64_t bv = sdesc_sw128(sbase + VT_OFF + (s >> 2) * VT_KB + (s & 3) * 32, 16, 1024);
        mma_tf32_ts(tbase + TM_U, tbase + TM_TB + s * 8, bv, idu, s > 0);
      }
      mma_commit(&misc->bar_2);
      if (t0 + C < t_end) {
        issue_tma(t0 + C);
        tma_out = true;
        tma_par = (it + 1) & 1u;
      }
    }
    if (!mbar_wait(&misc->bar_2, par)) misc->abort = 1;
    tc_fence_after();
    if (qd < 2) {  // token rows 0..63: U (16 columns per warp) stored as U^T (K-major)
      float u[16];
      tmem_ld16(tbase + lane_base + TM_U + ch * 16, u);
      const int r = qd * 32 + lane;
#pragma unroll
      for (int j = 0; j < 16; ++j) *f32at(sm, UT_OFF + sw128_off32(ch * 16 + j, r, UT_KB)) = u[j];
    }
    fence_proxy_async_smem();
    cta_sync();
    if (misc->abort) { ok = false; break; }
    // ================= round 3: Y = Kb^T U, O = X_q + tril(A_qk) U
    if (tid == 0) {
      const uint32_t idy = idesc_make(kFmtTF32, 128, 32, false, false);
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        const uint64_t b = sdesc_sw128(sbase + UT_OFF + (s >> 2) * UT_KB + (s & 3) * 32, 16, 1024);
        mma_tf32_ts(tbase + TM_Y, tbase + tm_kbt + s * 8, b, idy, s > 0);
        if (!pkg) mma_tf32_ts(tbase + TM_X, tbase + tma_a + s * 8, b, idy, 1);
      }
      mma_commit(&misc->bar_3);
    }
    // While round 3 runs: build the next chunk's operands (its loads were issued in round 2;
    // XA and KB are free, and its A and Kb^T go to the other TMEM buffers) and start its A.
    float rho2_next = rho2;
    if (t0 + C < t_end) {
      rho2_next = build(t0 + C, it + 1);
      fence_proxy_async_smem();
      cta_sync();
      if (tid == 0 && !misc->abort) issue_a(it + 1);
    }
    if (!mbar_wait(&misc->bar_3, par)) misc->abort = 1;
    tc_fence_after();
    if (qd >= 2 && !pkg && p.o) {  // output rows (Qh rows 64..127), 16 columns per warp
      float x[16];
      tmem_ld16(tbase + lane_base + TM_X + ch * 16, x);
      const int r = qd * 32 + lane - C;
      if (r < n) {
        __nv_bfloat16* o = (__nv_bfloat16*)p.o + ((int64_t)(t0 + r) * H + h) * DK + j0 + ch * 16;
#pragma unroll
        for (int j = 0; j < 16; j += 8) {
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
    {  // state: S = e^(2 rho) S + e^rho Y (lane c; 16 columns per warp)
      float s[16], y[16];
      tmem_ld16(tbase + lane_base + TM_S + ch * 16, s);
      tmem_ld16(tbase + lane_base + TM_Y + ch * 16, y);
#pragma unroll
      for (int j = 0; j < 16; ++j) s[j] = erho * fmaf(erho, s[j], y[j]);
      tmem_st16(tbase + lane_base + TM_S + ch * 16, s);
      tmem_st_wait();
    }
    rho2 = rho2_next;
    cta_sync();
    if (misc->abort) { ok = false; break; }
  }
  if (misc->abort) ok = false;
  // ---- exit state of this tile
  if (!ok) {
    // Let this CTA's in-flight MMAs and loads drain (bounded) before its shared memory and
    // TMEM are released.
    if (tid == 0) {
      if (p.status) atomicOr(p.status, KDA_STATUS_TIMEOUT);
      mma_commit(&misc->bar_drain);
      mbar_wait(&misc->bar_drain, 0, 100000000ull);
      if (tma_out) mbar_wait(&misc->bar_tma, tma_par, 100000000ull);
    }
  } else {
    float s[16];
    tmem_ld16(tbase + lane_base + TM_S + ch * 16, s);
    const int64_t sh = (int64_t)sidx * H + h;
    float* dst = nullptr;
    if (pkg) dst = mcols ? p.M + (sh * DK + c) * DK + j0 : p.D + (sh * DK + c) * DK + vcol0;
    else if (p.final_state) dst = p.final_state + (sh * DK + c) * DK + j0;
    if (dst) {
#pragma unroll
      for (int j = 0; j < 16; j += 4)
        *reinterpret_cast<float4*>(dst + ch * 16 + j) =
            make_float4(s[j], s[j + 1], s[j + 2], s[j + 3]);
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

// [T, H, d] (bf16, or fp32 when f32) viewed as a 3-D tensor (d, H, T); box (box_d, 1, 64).
bool make_map3(CUtensorMap* m, const void* ptr, int T, int H, int d, int box_d, bool swizzle,
               bool f32) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t es_bytes = f32 ? 4 : 2;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)(T > 0 ? T : 1)};
  cuuint64_t strides[2] = {(cuuint64_t)d * es_bytes, (cuuint64_t)H * d * es_bytes};
  cuuint32_t box[3] = {(cuuint32_t)box_d, 1, (cuuint32_t)C};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                   const_cast<void*>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
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

}  // namespace

bool chunk_tc_supported(const ChunkParams& p, kda_dtype dt) {
  return dt == KDA_BF16 && p.dk == 128 && p.dv == 128 && p.total_tokens > 0 && p.H % 4 == 0 &&
         ((uintptr_t)p.beta % 16) == 0 && encode_fn() != nullptr;
}

kda_status launch_chunk_tc(const ChunkParams& p, kda_dtype dt, cudaStream_t s) {
  (void)dt;
  if (p.n_ranges == 0) return KDA_OK;
  CUtensorMap mq, mk, mv, mg, mb;
  const void* qp = p.q ? p.q : p.k;
  if (!make_map3(&mq, qp, p.total_tokens, p.H, 128, 64, true, false) ||
      !make_map3(&mk, p.k, p.total_tokens, p.H, 128, 64, true, false) ||
      !make_map3(&mv, p.v, p.total_tokens, p.H, 128, TW, false, false) ||
      !make_map3(&mg, p.g, p.total_tokens, p.H, 128, 128, false, true) ||
      !make_map_beta(&mb, p.beta, p.total_tokens, p.H))
    return set_error(KDA_ERR_CUDA, "tensor-core chunk kernel: cuTensorMapEncodeTiled failed");
  cudaError_t e = cudaFuncSetAttribute(chunk_tc_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess)
    return set_error(KDA_ERR_CUDA, std::string("tensor-core chunk kernel attribute: ") +
                                       cudaGetErrorString(e));
  const int cols = p.package ? (p.dk + p.dv) : p.dv;
  dim3 grid(cols / TW, p.H, p.n_ranges);
  chunk_tc_kernel<<<grid, kThreads, SMEM_BYTES, s>>>(p, mq, mk, mv, mg, mb);
  count_launches(1);
  return check_launch("tensor-core chunk kernel");
}

}  // namespace kda
