// Chunked KDA pass on CUDA cores (fp32 FFMA): the exact-arithmetic path (fp32 inputs) and
// the package/replay fallback for shapes the tensor-core kernel does not take.
//
// Chunk algebra (per range, head, 64-token chunk; S_0 = state entering the chunk).
// The pages name the chunked FlashKDA prefill (kern PR #44; pegainfer PR #970, "same segment
// walk, same chunk step") but do not write its algebra; the form below is the standard
// WY/UT rearrangement of the gated delta rule, restated here from the recurrence:
//   gamma_r = sum_{i<=r} g_i (per key channel), rho = gamma_C / 2 (log-midpoint of the chunk)
//   Kh_r = k_r * exp(gamma_r - rho),  Qh_r = q_r * exp(gamma_r - rho),
//   Kb_r = k_r * exp(rho - gamma_r)
//   A_kk[r,i] = beta_r Kh_r . Kb_i  (i < r),     A_qk[r,i] = Qh_r . Kb_i  (i <= r)
//   T = (I + A_kk)^-1,  W = T diag(beta) Kh,  Ut = T diag(beta) V
//   Sh = Diag(exp(rho)) S_0            (the chunk's state in the midpoint frame)
//   U = Ut - W Sh,   O = scale (Qh Sh + A_qk U),
//   S_C = Diag(exp(gamma_C - rho)) Sh + Kb'^T U,   Kb'_r = k_r * exp(gamma_C - gamma_r)
// Every exponent stays within +-|gamma_C|/2, so a channel that decays by at most 160 nats
// over the chunk never overflows fp32. A channel that decays more ("strong") takes rho = 0
// and Kb = 0, so it has no share in the Kh Kb^T products; its share of A_kk and A_qk is added
// exactly, each pairwise factor exp(gamma_r - gamma_i) = a_{i+1} ... a_r built as a product
// of the per-token decays a = exp(g) <= 1 (no overflow, and no loss to the cancellation of
// large cumulative sums). Kb' comes from suffix sums of g for the same reason.
//
// A CTA owns one (range, head, 32-column tile) and walks the range's chunks in order; the
// tile's state columns stay in shared memory. Columns are independent in the recurrence, so
// tiles never communicate; the K-side work (A, T, W) is recomputed per tile.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int C = kChunk;
constexpr int TW = 32;        // state columns per CTA
constexpr int LT = TW + 1;    // padded stride of 32-wide tiles
constexpr int LC = C + 1;     // padded stride of 64-wide tiles
constexpr int kThreads = 256;

template <int DK>
constexpr size_t simt_smem_floats() {
  return (size_t)4 * C * (DK + 1) + 3 * (size_t)C * LC + 2 * (size_t)C * LT +
         (size_t)DK * LT + 3 * DK + C;
}

template <int DK, class T>
__global__ void __launch_bounds__(kThreads, 1) chunk_simt_kernel(ChunkParams p) {
  constexpr int LDK = DK + 1;
  constexpr int DV = DK;
  extern __shared__ float smem[];
  float* Qh = smem;               // [C][LDK]
  float* Kh = Qh + C * LDK;       // [C][LDK]
  float* Kb = Kh + C * LDK;       // [C][LDK]
  float* Gw = Kb + C * LDK;       // [C][LDK]  gamma, then W
  float* Akk = Gw + C * LDK;      // [C][LC]   A_kk, then T diag(beta)
  float* Aqk = Akk + C * LC;      // [C][LC]
  float* X = Aqk + C * LC;        // [C][LC]   (I + A_kk)^-1
  float* Vs = X + C * LC;         // [C][LT]
  float* Us = Vs + C * LT;        // [C][LT]   Ut, then U
  float* Ss = Us + C * LT;        // [DK][LT]  state tile
  float* rho = Ss + DK * LT;      // [DK]
  float* gC = rho + DK;           // [DK]
  float* bs = gC + DK;            // [C]
  int* strong = reinterpret_cast<int*>(bs + C);  // [DK] channel decays beyond the frame

  const int tid = threadIdx.x;
  const int tile = blockIdx.x, h = blockIdx.y, sidx = blockIdx.z;
  const int H = p.H;
  int t_begin = 0, t_end = p.total_tokens;
  if (p.offsets) {
    t_begin = p.offsets[sidx];
    t_end = p.offsets[sidx + 1];
    if (t_end < t_begin || t_begin < 0 || t_end > p.total_tokens) {
      if (tid == 0 && p.status) atomicOr(p.status, KDA_STATUS_BAD_OFFSETS);
      t_end = t_begin;  // treat as empty
    }
  }
  const bool pkg = p.package != 0;
  const int j0 = tile * TW;                   // column in the (augmented) column space
  const bool mcols = pkg && j0 < DK;          // identity-initialised, zero-valued columns
  const int vcol0 = pkg ? j0 - DK : j0;       // value column of this tile's first column
  const T* q = (const T*)p.q;
  const T* k = (const T*)p.k;
  const T* v = (const T*)p.v;

  for (int idx = tid; idx < DK * TW; idx += kThreads) {
    const int c = idx / TW, j = idx - c * TW;
    float x = 0.0f;
    if (pkg) x = (mcols && c == j0 + j) ? 1.0f : 0.0f;
    else if (p.init) x = p.init[(((int64_t)sidx * H + h) * DK + c) * DV + j0 + j];
    Ss[c * LT + j] = x;
  }

  for (int t0 = t_begin; t0 < t_end; t0 += C) {
    const int n = min(C, t_end - t0);
    __syncthreads();
    // ---- load g (zero past the range), beta, and the value tile
    for (int idx = tid; idx < C * DK; idx += kThreads) {
      const int r = idx / DK, c = idx - r * DK;
      Gw[r * LDK + c] = (r < n) ? p.g[((int64_t)(t0 + r) * H + h) * DK + c] : 0.0f;
    }
    if (tid < C) bs[tid] = (tid < n) ? p.beta[(int64_t)(t0 + tid) * H + h] : 0.0f;
    for (int idx = tid; idx < C * TW; idx += kThreads) {
      const int r = idx / TW, j = idx - r * TW;
      float x = 0.0f;
      if (r < n && !mcols) x = ld_elem(v, ((int64_t)(t0 + r) * H + h) * DV + vcol0 + j);
      Vs[r * LT + j] = x;
    }
    __syncthreads();
    // ---- cumulative log-decay per channel
    bool my_strong = false;
    if (tid < DK) {
      float acc = 0.0f;
      for (int r = 0; r < C; ++r) {
        acc += Gw[r * LDK + tid];
        Gw[r * LDK + tid] = acc;
      }
      gC[tid] = acc;
      my_strong = !(acc >= -kMaxChunkDecay);
      strong[tid] = my_strong;
      rho[tid] = my_strong ? 0.0f : 0.5f * acc;
    }
    const bool any_strong = __syncthreads_or(my_strong) != 0;
    // ---- midpoint-frame operands and the state in the midpoint frame
    for (int idx = tid; idx < C * DK; idx += kThreads) {
      const int r = idx / DK, c = idx - r * DK;
      const float x = Gw[r * LDK + c] - rho[c];
      const float e1 = expf(x);
      const int64_t e = ((int64_t)(t0 + r) * H + h) * DK + c;
      const float kv = (r < n) ? ld_elem(k, e) : 0.0f;
      Kh[r * LDK + c] = kv * e1;
      Kb[r * LDK + c] = strong[c] ? 0.0f : kv * expf(-x);
      if (!pkg) Qh[r * LDK + c] = ((r < n) ? ld_elem(q, e) : 0.0f) * e1;
    }
    for (int idx = tid; idx < DK * TW; idx += kThreads) {
      const int c = idx / TW, j = idx - c * TW;
      Ss[c * LT + j] *= expf(rho[c]);
    }
    __syncthreads();
    // ---- intra-chunk products
    for (int idx = tid; idx < C * C; idx += kThreads) {
      const int r = idx / C, i = idx - r * C;
      float akk = 0.0f, aqk = 0.0f;
      if (i <= r) {
        for (int c = 0; c < DK; ++c) {
          const float kb = Kb[i * LDK + c];
          akk = fmaf(Kh[r * LDK + c], kb, akk);
          if (!pkg) aqk = fmaf(Qh[r * LDK + c], kb, aqk);
        }
      }
      Akk[r * LC + i] = (i < r) ? bs[r] * akk : 0.0f;
      Aqk[r * LC + i] = (i <= r) ? aqk : 0.0f;
      X[r * LC + i] = (i == r) ? 1.0f : 0.0f;
    }
    __syncthreads();
    // ---- the strong channels' exact shares: thread r owns row r of A_kk and A_qk and runs
    // i from r down to 0 with f = exp(gamma_r - gamma_i) = f(i + 1) * a_{i + 1}
    if (any_strong) {
      if (tid < n) {
        const int r = tid;
        for (int c = 0; c < DK; ++c) {
          if (!strong[c]) continue;
          const int64_t er = ((int64_t)(t0 + r) * H + h) * DK + c;
          const float kr = ld_elem(k, er);
          const float qr = pkg ? 0.0f : ld_elem(q, er);
          float f = 1.0f;
          for (int i = r; i >= 0; --i) {
            const int64_t ei = ((int64_t)(t0 + i) * H + h) * DK + c;
            const float ki = ld_elem(k, ei);
            if (i < r) Akk[r * LC + i] = fmaf(bs[r] * kr * ki, f, Akk[r * LC + i]);
            if (!pkg) Aqk[r * LC + i] = fmaf(qr * ki, f, Aqk[r * LC + i]);
            f *= expf(p.g[ei]);
          }
        }
      }
      __syncthreads();
    }
    // ---- Kb' = k exp(gamma_C - gamma_r) (Kb is read no more): suffix sums of g per channel
    if (tid < DK) {
      float suf = 0.0f;  // gamma_C - gamma_r = sum of g over the chunk's tokens after r
      for (int r = C - 1; r >= 0; --r) {
        const int64_t e = ((int64_t)(t0 + r) * H + h) * DK + tid;
        const bool valid = r < n;
        Kb[r * LDK + tid] = valid ? ld_elem(k, e) * expf(suf) : 0.0f;
        if (valid) suf += p.g[e];
      }
    }
    __syncthreads();
    // ---- X = (I + A_kk)^-1 by right-looking forward substitution over columns l
    for (int l = 0; l < C - 1; ++l) {
      const int rows = C - 1 - l, cols = l + 1;
      for (int idx = tid; idx < rows * cols; idx += kThreads) {
        const int rr = l + 1 + idx / cols, i = idx % cols;
        X[rr * LC + i] -= Akk[rr * LC + l] * X[l * LC + i];
      }
      __syncthreads();
    }
    // T diag(beta) into Akk
    for (int idx = tid; idx < C * C; idx += kThreads) {
      const int r = idx / C, i = idx - r * C;
      Akk[r * LC + i] = (i <= r) ? X[r * LC + i] * bs[i] : 0.0f;
    }
    __syncthreads();
    // ---- W = T diag(beta) Kh (into Gw), Ut = T diag(beta) V (into Us)
    for (int idx = tid; idx < C * DK; idx += kThreads) {
      const int r = idx / DK, c = idx - r * DK;
      float acc = 0.0f;
      for (int i = 0; i <= r; ++i) acc = fmaf(Akk[r * LC + i], Kh[i * LDK + c], acc);
      Gw[r * LDK + c] = acc;
    }
    for (int idx = tid; idx < C * TW; idx += kThreads) {
      const int r = idx / TW, j = idx - r * TW;
      float acc = 0.0f;
      if (!mcols)
        for (int i = 0; i <= r; ++i) acc = fmaf(Akk[r * LC + i], Vs[i * LT + j], acc);
      Us[r * LT + j] = acc;
    }
    __syncthreads();
    // ---- U = Ut - W Sh
    for (int idx = tid; idx < C * TW; idx += kThreads) {
      const int r = idx / TW, j = idx - r * TW;
      float acc = Us[r * LT + j];
      for (int c = 0; c < DK; ++c) acc = fmaf(-Gw[r * LDK + c], Ss[c * LT + j], acc);
      Us[r * LT + j] = acc;
    }
    __syncthreads();
    // ---- O = scale (Qh Sh + A_qk U)
    if (!pkg && p.o) {
      T* o = (T*)p.o;
      for (int idx = tid; idx < C * TW; idx += kThreads) {
        const int r = idx / TW, j = idx - r * TW;
        if (r >= n) continue;
        float acc = 0.0f;
        for (int c = 0; c < DK; ++c) acc = fmaf(Qh[r * LDK + c], Ss[c * LT + j], acc);
        for (int i = 0; i <= r; ++i) acc = fmaf(Aqk[r * LC + i], Us[i * LT + j], acc);
        st_elem(o, ((int64_t)(t0 + r) * H + h) * DV + j0 + j, p.scale * acc);
      }
      __syncthreads();
    }
    // ---- S_C = Diag(exp(gamma_C - rho)) Sh + Kb'^T U
    for (int idx = tid; idx < DK * TW; idx += kThreads) {
      const int c = idx / TW, j = idx - c * TW;
      float acc = Ss[c * LT + j] * expf(gC[c] - rho[c]);
      for (int i = 0; i < C; ++i) acc = fmaf(Kb[i * LDK + c], Us[i * LT + j], acc);
      Ss[c * LT + j] = acc;
    }
  }
  __syncthreads();
  // ---- exit state of this tile
  for (int idx = tid; idx < DK * TW; idx += kThreads) {
    const int c = idx / TW, j = idx - c * TW;
    const float x = Ss[c * LT + j];
    const int64_t sh = (int64_t)sidx * H + h;
    if (pkg) {
      if (mcols) p.M[(sh * DK + c) * DK + j0 + j] = x;
      else p.D[(sh * DK + c) * DV + vcol0 + j] = x;
    } else if (p.final_state) {
      p.final_state[(sh * DK + c) * DV + j0 + j] = x;
    }
  }
}

template <int DK, class T>
kda_status launch_dk(const ChunkParams& p, cudaStream_t s) {
  const size_t bytes = simt_smem_floats<DK>() * sizeof(float);
  auto kern = chunk_simt_kernel<DK, T>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)bytes);
  if (e != cudaSuccess)
    return set_error(KDA_ERR_CUDA, std::string("chunk kernel attribute: ") +
                                       cudaGetErrorString(e));
  const int cols = p.package ? (p.dk + p.dv) : p.dv;
  dim3 grid(cols / TW, p.H, p.n_ranges);
  kern<<<grid, kThreads, bytes, s>>>(p);
  count_launches(1);
  return check_launch("chunk kernel (CUDA cores)");
}

}  // namespace

kda_status launch_chunk_simt(const ChunkParams& p, kda_dtype dt, cudaStream_t s) {
  if (p.n_ranges == 0) return KDA_OK;
  if (p.dk == 128) return dt == KDA_BF16 ? launch_dk<128, __nv_bfloat16>(p, s)
                                         : launch_dk<128, float>(p, s);
  if (p.dk == 64) return dt == KDA_BF16 ? launch_dk<64, __nv_bfloat16>(p, s)
                                        : launch_dk<64, float>(p, s);
  return set_error(KDA_ERR_UNSUPPORTED, "chunk kernel: dk must be 64 or 128");
}

}  // namespace kda
