// One-token KDA decode over a slot-addressed fp32 state pool (in place).
//
// For batch row b and head h, with S = pool[slot_ids[b], h] (dk x dv, row = key channel):
//     x = (Diag(a) S)^T k,  y = (Diag(a) S)^T q,  u = v - x,
//     S' = Diag(a) S + beta k u^T,   o = scale (y + beta (q.k) u)
// which is S' = (I - beta k k^T) Diag(a) S + beta k v^T and o = scale S'^T q, with one read
// and one write of S. Source: ATOM PR #2709 ("feat(kimi-k3): PP8 prefill for P/D serving -
// KDA state under PP"), decode through slot-indexed state tables.
//
// The pass is HBM-bound (64 KiB read + 64 KiB written per (row, head) at d = 128), so the
// kernel is laid out for bandwidth: one CTA per (row, head); warp w owns dk/8 consecutive
// state rows and lane l owns dv/32 consecutive columns, so each warp moves whole 512-byte
// rows with 16-byte vector accesses, all of a CTA's loads are issued before any reduction,
// and the state streams with evict-first cache hints. The two column reductions over the key
// channels run as in-register partial sums, one shared-memory exchange between the 8 warps.
#include "kda_internal.cuh"

namespace kda {
namespace {

// 8 warps per CTA (16 state rows each at dk = 128) and 2 CTAs per SM: 16 resident warps keep
// 16 x 16 x 512 B = 128 KiB of state loads in flight per SM. (16 warps of 8 rows measured
// 3% slower.)
constexpr int kWarps = 8;

template <int DK, int DV, class T>
__global__ void __launch_bounds__(kWarps * 32, 2)
decode_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
              const float* __restrict__ g, const float* __restrict__ beta,
              const int32_t* __restrict__ slot_ids, float* __restrict__ pool, int64_t n_slots,
              int H, float scale, T* __restrict__ o, uint32_t* status) {
  constexpr int RPW = DK / kWarps;  // state rows per warp
  constexpr int CPL = DV / 32;      // columns per lane (4 or 2)
  static_assert(CPL == 4 || CPL == 2, "dv must be 64 or 128");
  const int bh = blockIdx.x;
  const int b = bh / H, h = bh - b * H;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t tok = (int64_t)b * H + h;
  const int slot = slot_ids[b];

  __shared__ float red_x[kWarps][DV];
  __shared__ float red_y[kWarps][DV];
  __shared__ float qk_part[kWarps];
  __shared__ float tot_x[DV], tot_y[DV];

  if (slot < 0 || (int64_t)slot >= n_slots) {
    if ((int64_t)slot >= n_slots && threadIdx.x == 0 && h == 0 && status)
      atomicOr(status, KDA_STATUS_BAD_SLOT);
    for (int j = threadIdx.x; j < DV; j += blockDim.x) st_elem(o, tok * DV + j, 0.0f);
    return;
  }

  float* S = pool + ((int64_t)slot * H + h) * (int64_t)DK * DV;
  const int r0 = warp * RPW;
  const int c0 = lane * CPL;

  // Issue every state load of this thread first (RPW independent vector loads).
  float st[RPW][CPL];
#pragma unroll
  for (int i = 0; i < RPW; ++i) {
    const float* src = S + (int64_t)(r0 + i) * DV + c0;
    if constexpr (CPL == 4) {
      float4 t4 = __ldcs(reinterpret_cast<const float4*>(src));
      st[i][0] = t4.x; st[i][1] = t4.y; st[i][2] = t4.z; st[i][3] = t4.w;
    } else {
      float2 t2 = __ldcs(reinterpret_cast<const float2*>(src));
      st[i][0] = t2.x; st[i][1] = t2.y;
    }
  }

  // Per-row decay and key/query entries of this warp's rows (lanes read the same words).
  float a[RPW], kr[RPW], qr[RPW];
  float qk = 0.0f;
#pragma unroll
  for (int i = 0; i < RPW; ++i) {
    const int64_t e = tok * DK + r0 + i;
    a[i] = __expf(g[e]);
    kr[i] = ld_elem(k, e);
    qr[i] = ld_elem(q, e);
    qk = fmaf(qr[i], kr[i], qk);
  }

  // Decay in registers, then partial column sums over this warp's rows.
  float px[CPL], py[CPL];
#pragma unroll
  for (int j = 0; j < CPL; ++j) { px[j] = 0.0f; py[j] = 0.0f; }
#pragma unroll
  for (int i = 0; i < RPW; ++i) {
#pragma unroll
    for (int j = 0; j < CPL; ++j) {
      st[i][j] *= a[i];
      px[j] = fmaf(kr[i], st[i][j], px[j]);
      py[j] = fmaf(qr[i], st[i][j], py[j]);
    }
  }
#pragma unroll
  for (int j = 0; j < CPL; ++j) {
    red_x[warp][c0 + j] = px[j];
    red_y[warp][c0 + j] = py[j];
  }
  if (lane == 0) qk_part[warp] = qk;
  __syncthreads();
  // column totals over the warps: one thread per (column, x|y)
  if (threadIdx.x < 2 * DV) {
    const int col = threadIdx.x % DV;
    float s = 0.0f;
    if (threadIdx.x < DV) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) s += red_x[w][col];
      tot_x[col] = s;
    } else {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) s += red_y[w][col];
      tot_y[col] = s;
    }
  }
  __syncthreads();

  const float bt = beta[tok];
  float qk_all = 0.0f;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) qk_all += qk_part[w];
  float u[CPL];
#pragma unroll
  for (int j = 0; j < CPL; ++j) {
    const float x = tot_x[c0 + j], y = tot_y[c0 + j];
    u[j] = ld_elem(v, tok * DV + c0 + j) - x;
    if (warp == 0) st_elem(o, tok * DV + c0 + j, scale * (y + bt * qk_all * u[j]));
  }

  // S' = Diag(a) S + beta k u^T, written back in place.
#pragma unroll
  for (int i = 0; i < RPW; ++i) {
    const float bk = bt * kr[i];
    float* dst = S + (int64_t)(r0 + i) * DV + c0;
    if constexpr (CPL == 4) {
      float4 t4 = make_float4(fmaf(bk, u[0], st[i][0]), fmaf(bk, u[1], st[i][1]),
                              fmaf(bk, u[2], st[i][2]), fmaf(bk, u[3], st[i][3]));
      __stcs(reinterpret_cast<float4*>(dst), t4);
    } else {
      float2 t2 = make_float2(fmaf(bk, u[0], st[i][0]), fmaf(bk, u[1], st[i][1]));
      __stcs(reinterpret_cast<float2*>(dst), t2);
    }
  }
}

// Verify window with a state fork: row b reads its state from slot read_slots[b], runs the
// W tokens of its window (token b*W + j) and stores the state after token j into slot
// write_slots[b*W + j] (nothing for a negative id), so that a caller that accepts n tokens
// resumes from column n - 1's snapshot. Source: ATOM PR #2709 ("feat(kimi-k3): PP8 prefill
// for P/D serving - KDA state under PP"), commits "read a forked state through the kernels'
// read-side index" (a fork is read through a read index instead of being copied onto the
// write slot) and the verify-window fix of the same page (a window keeps one state column per
// position and the next step starts from the last accepted one). With KDA_DECODE_BETA_LOGIT
// the write strength is sigmoid(beta), as in the sigmoid-gated delta-rule update named in
// the same commit.
//
// Same layout as decode_kernel: one CTA per (row, head), state in registers for the whole
// window (one read of 64 KiB at d = 128, then one streamed 64 KiB store per stored column).
// The window's inputs are staged once in shared memory (exp(g), k, q, v, beta), so each
// token's per-row operands are shared-memory broadcasts instead of dependent global loads.
template <int DK, int DV, class T>
__global__ void __launch_bounds__(kWarps * 32, 2)
decode_window_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                     const float* __restrict__ g, const float* __restrict__ beta,
                     unsigned flags, const int32_t* __restrict__ read_slots,
                     const int32_t* __restrict__ write_slots, float* __restrict__ pool,
                     int64_t n_slots, int H, int W, float scale, T* __restrict__ o,
                     uint32_t* status) {
  constexpr int RPW = DK / kWarps;
  constexpr int CPL = DV / 32;
  static_assert(CPL == 4 || CPL == 2, "dv must be 64 or 128");
  const int bh = blockIdx.x;
  const int b = bh / H, h = bh - b * H;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r0 = warp * RPW;
  const int c0 = lane * CPL;

  extern __shared__ float win[];      // [W][DK] exp(g), k, q; [W][DV] v; [W] beta
  float* s_a = win;
  float* s_k = s_a + W * DK;
  float* s_q = s_k + W * DK;
  float* s_v = s_q + W * DK;
  float* s_b = s_v + W * DV;
  __shared__ float red_x[kWarps][DV];
  __shared__ float red_y[kWarps][DV];
  __shared__ float qk_part[2][kWarps];  // by token parity: the next token's partials may be
                                        // written while slower warps still read these
  __shared__ float tot_x[DV], tot_y[DV];

  const int slot = read_slots[b];
  if (slot < 0 || (int64_t)slot >= n_slots) {
    if ((int64_t)slot >= n_slots && threadIdx.x == 0 && h == 0 && status)
      atomicOr(status, KDA_STATUS_BAD_SLOT);
    for (int i = threadIdx.x; i < W * DV; i += blockDim.x) {
      const int j = i / DV, c = i - j * DV;
      st_elem(o, ((int64_t)(b * W + j) * H + h) * DV + c, 0.0f);
    }
    return;
  }

  const float* S = pool + ((int64_t)slot * H + h) * (int64_t)DK * DV;
  float st[RPW][CPL];
#pragma unroll
  for (int i = 0; i < RPW; ++i) {
    const float* src = S + (int64_t)(r0 + i) * DV + c0;
    if constexpr (CPL == 4) {
      float4 t4 = __ldcs(reinterpret_cast<const float4*>(src));
      st[i][0] = t4.x; st[i][1] = t4.y; st[i][2] = t4.z; st[i][3] = t4.w;
    } else {
      float2 t2 = __ldcs(reinterpret_cast<const float2*>(src));
      st[i][0] = t2.x; st[i][1] = t2.y;
    }
  }

  // stage the window's inputs (token-major rows: token b*W + j, head h)
  for (int i = threadIdx.x; i < W * DK; i += blockDim.x) {
    const int j = i / DK, c = i - j * DK;
    const int64_t e = ((int64_t)(b * W + j) * H + h) * DK + c;
    s_a[i] = __expf(g[e]);
    s_k[i] = ld_elem(k, e);
    s_q[i] = ld_elem(q, e);
  }
  for (int i = threadIdx.x; i < W * DV; i += blockDim.x) {
    const int j = i / DV, c = i - j * DV;
    s_v[i] = ld_elem(v, ((int64_t)(b * W + j) * H + h) * DV + c);
  }
  for (int j = threadIdx.x; j < W; j += blockDim.x) {
    const float x = beta[(int64_t)(b * W + j) * H + h];
    s_b[j] = (flags & KDA_DECODE_BETA_LOGIT) ? 1.0f / (1.0f + expf(-x)) : x;
  }
  __syncthreads();

  for (int j = 0; j < W; ++j) {
    const float* a = s_a + j * DK + r0;
    const float* kr = s_k + j * DK + r0;
    const float* qr = s_q + j * DK + r0;
    float qk = 0.0f;
#pragma unroll
    for (int i = 0; i < RPW; ++i) qk = fmaf(qr[i], kr[i], qk);
    float px[CPL], py[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c) { px[c] = 0.0f; py[c] = 0.0f; }
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
#pragma unroll
      for (int c = 0; c < CPL; ++c) {
        st[i][c] *= a[i];
        px[c] = fmaf(kr[i], st[i][c], px[c]);
        py[c] = fmaf(qr[i], st[i][c], py[c]);
      }
    }
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
      red_x[warp][c0 + c] = px[c];
      red_y[warp][c0 + c] = py[c];
    }
    if (lane == 0) qk_part[j & 1][warp] = qk;
    __syncthreads();
    if (threadIdx.x < 2 * DV) {
      const int col = threadIdx.x % DV;
      float s = 0.0f;
      if (threadIdx.x < DV) {
#pragma unroll
        for (int w = 0; w < kWarps; ++w) s += red_x[w][col];
        tot_x[col] = s;
      } else {
#pragma unroll
        for (int w = 0; w < kWarps; ++w) s += red_y[w][col];
        tot_y[col] = s;
      }
    }
    __syncthreads();

    const float bt = s_b[j];
    float qk_all = 0.0f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) qk_all += qk_part[j & 1][w];
    const int64_t tok = (int64_t)(b * W + j) * H + h;
    float u[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
      const float x = tot_x[c0 + c], y = tot_y[c0 + c];
      u[c] = s_v[j * DV + c0 + c] - x;
      if (warp == 0) st_elem(o, tok * DV + c0 + c, scale * (y + bt * qk_all * u[c]));
    }
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
      const float bk = bt * kr[i];
#pragma unroll
      for (int c = 0; c < CPL; ++c) st[i][c] = fmaf(bk, u[c], st[i][c]);
    }

    // this column's snapshot
    const int ws = write_slots[(int64_t)b * W + j];
    if ((int64_t)ws >= n_slots) {
      if (threadIdx.x == 0 && h == 0 && status) atomicOr(status, KDA_STATUS_BAD_SLOT);
    } else if (ws >= 0) {
      float* D = pool + ((int64_t)ws * H + h) * (int64_t)DK * DV;
#pragma unroll
      for (int i = 0; i < RPW; ++i) {
        float* dst = D + (int64_t)(r0 + i) * DV + c0;
        if constexpr (CPL == 4)
          __stcs(reinterpret_cast<float4*>(dst), make_float4(st[i][0], st[i][1], st[i][2], st[i][3]));
        else
          __stcs(reinterpret_cast<float2*>(dst), make_float2(st[i][0], st[i][1]));
      }
    }
  }
}

template <int DK, int DV>
constexpr size_t window_smem_bytes(int W) {
  return (size_t)W * (3 * DK + DV + 1) * sizeof(float);
}

template <int DK, int DV, class T>
kda_status launch_window_t(int batch, int window, int H, float scale, const void* q,
                           const void* k, const void* v, const float* g, const float* beta,
                           unsigned flags, const int32_t* read_slots,
                           const int32_t* write_slots, float* pool, int64_t n_slots, void* o,
                           uint32_t* status, cudaStream_t s) {
  dim3 grid((unsigned)batch * (unsigned)H);
  decode_window_kernel<DK, DV, T><<<grid, kWarps * 32, window_smem_bytes<DK, DV>(window), s>>>(
      (const T*)q, (const T*)k, (const T*)v, g, beta, flags, read_slots, write_slots, pool,
      n_slots, H, window, scale, (T*)o, status);
  count_launches(1);
  return check_launch("kda_decode_window");
}

template <int DK, int DV, class T>
void launch_t(int batch, int H, float scale, const void* q, const void* k, const void* v,
              const float* g, const float* beta, const int32_t* slots, float* pool,
              int64_t n_slots, void* o, uint32_t* status, cudaStream_t s) {
  dim3 grid((unsigned)batch * (unsigned)H);
  decode_kernel<DK, DV, T><<<grid, kWarps * 32, 0, s>>>(
      (const T*)q, (const T*)k, (const T*)v, g, beta, slots, pool, n_slots, H, scale, (T*)o,
      status);
}

}  // namespace

kda_status launch_decode(kda_dtype dt, int batch, int H, int dk, int dv, float scale,
                         const void* q, const void* k, const void* v, const float* g,
                         const float* beta, const int32_t* slot_ids, float* pool,
                         int64_t n_slots, void* o, uint32_t* status, cudaStream_t s) {
  if (batch == 0) return KDA_OK;
  if (dk == 128 && dv == 128) {
    if (dt == KDA_BF16)
      launch_t<128, 128, __nv_bfloat16>(batch, H, scale, q, k, v, g, beta, slot_ids, pool,
                                        n_slots, o, status, s);
    else
      launch_t<128, 128, float>(batch, H, scale, q, k, v, g, beta, slot_ids, pool, n_slots, o,
                                status, s);
  } else if (dk == 64 && dv == 64) {
    if (dt == KDA_BF16)
      launch_t<64, 64, __nv_bfloat16>(batch, H, scale, q, k, v, g, beta, slot_ids, pool,
                                      n_slots, o, status, s);
    else
      launch_t<64, 64, float>(batch, H, scale, q, k, v, g, beta, slot_ids, pool, n_slots, o,
                              status, s);
  } else {
    return set_error(KDA_ERR_UNSUPPORTED, "kda_decode_step: dk = dv must be 64 or 128");
  }
  count_launches(1);
  return check_launch("kda_decode_step");
}

kda_status launch_decode_window(kda_dtype dt, int batch, int window, int H, int dk, int dv,
                                float scale, const void* q, const void* k, const void* v,
                                const float* g, const float* beta, unsigned flags,
                                const int32_t* read_slots, const int32_t* write_slots,
                                float* pool, int64_t n_slots, void* o, uint32_t* status,
                                cudaStream_t s) {
  if (batch == 0 || window == 0) return KDA_OK;
  if (dk == 128 && dv == 128) {
    if (dt == KDA_BF16)
      return launch_window_t<128, 128, __nv_bfloat16>(batch, window, H, scale, q, k, v, g, beta,
                                                      flags, read_slots, write_slots, pool,
                                                      n_slots, o, status, s);
    return launch_window_t<128, 128, float>(batch, window, H, scale, q, k, v, g, beta, flags,
                                            read_slots, write_slots, pool, n_slots, o, status,
                                            s);
  }
  if (dk == 64 && dv == 64) {
    if (dt == KDA_BF16)
      return launch_window_t<64, 64, __nv_bfloat16>(batch, window, H, scale, q, k, v, g, beta,
                                                    flags, read_slots, write_slots, pool,
                                                    n_slots, o, status, s);
    return launch_window_t<64, 64, float>(batch, window, H, scale, q, k, v, g, beta, flags,
                                          read_slots, write_slots, pool, n_slots, o, status, s);
  }
  return set_error(KDA_ERR_UNSUPPORTED, "kda_decode_window: dk = dv must be 64 or 128");
}

}  // namespace kda
