// KDA decode over a slot-addressed fp32 state pool: one token per row (kda_decode_step, in
// place), or a verify window of W tokens per row with a state fork (kda_decode_window).
//
// Per token, for batch row b and head h, with S the row's current state (dk x dv, row = key
// channel):
//     x = (Diag(a) S)^T k,  y = (Diag(a) S)^T q,  u = v - x,
//     S' = Diag(a) S + beta k u^T,   o = scale (y + beta (q.k) u)
// which is S' = (I - beta k k^T) Diag(a) S + beta k v^T and o = scale S'^T q, with one read
// and one write of S. Source: ATOM PR #2709 ("feat(kimi-k3): PP8 prefill for P/D serving -
// KDA state under PP"), decode through slot-indexed state tables.
//
// Verify windows: row b reads its state from slot read_slots[b], runs the W tokens of its
// window (token b*W + j) and stores the state after token j into slot write_slots[b*W + j]
// (nothing for a negative id), so that a caller that accepts n tokens resumes from column
// n - 1's snapshot. Source: the same page, commits "read a forked state through the kernels'
// read-side index" (a fork is read through a read index instead of being copied onto the write
// slot) and the verify-window fix (a window keeps one state column per position and the next
// step starts from the last accepted one). With KDA_DECODE_BETA_LOGIT the write strength is
// sigmoid(beta), as in the sigmoid-gated delta-rule update named in the same commit. The
// one-token decode step is the window W = 1 with the write slot equal to the read slot.
//
// The pass is HBM-bound ((1 + W) x 64 KiB of state per (row, head) at d = 128), so the kernel
// is laid out for bandwidth. Every state column evolves on its own (u, o and the update of
// column j read only column j and per-row scalars), so a CTA owns one (row, head, 64-column
// half) and keeps its 32 KiB of state in registers for the whole window: 8 warps own dk/8
// consecutive state rows each and lane l two consecutive columns, so each warp moves
// 256-byte row segments with 8-byte accesses and evict-first hints, and at 64 registers a
// thread 4 CTAs (32 warps) fit on an SM. (One CTA per (row, head) with all 128 columns held 2
// CTAs per SM and measured 13% slower on 4-token windows, 1.4% on single tokens.) The state is
// read once; the window's inputs (exp(g), k, q, this half's v, beta) are staged once in shared
// memory, so each token's per-row operands are broadcasts; the two column reductions over the
// key channels run as in-register partial sums and one shared-memory exchange between the
// warps; each stored column is one streamed store of the registers. Both halves of a (row,
// head) compute the same q.k and column sums in the same order, so the split changes no bit.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kWarps = 8;
constexpr int kCols = 64;  // state columns per CTA

template <int DK, int DV, class T>
__global__ void __launch_bounds__(kWarps * 32, 4)
decode_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
              const float* __restrict__ g, const float* __restrict__ beta, unsigned flags,
              const int32_t* __restrict__ read_slots, const int32_t* __restrict__ write_slots,
              float* __restrict__ pool, int64_t n_slots, int H, int W, float scale,
              T* __restrict__ o, uint32_t* status) {
  constexpr int NC = DV < kCols ? DV : kCols;
  constexpr int NSPLIT = DV / NC;
  constexpr int RPW = DK / kWarps;  // state rows per warp
  constexpr int CPL = NC / 32;      // columns per lane
  static_assert(CPL == 2, "a lane owns two columns");
  const int part = blockIdx.x % NSPLIT;
  const int bh = blockIdx.x / NSPLIT;
  const int b = bh / H, h = bh - b * H;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r0 = warp * RPW;
  const int c0 = lane * CPL;         // column within this CTA's half
  const int cg = part * NC + c0;     // column of the state

  extern __shared__ float win[];     // [W][DK] exp(g), k, q; [W][NC] v; [W] beta
  float* s_a = win;
  float* s_k = s_a + W * DK;
  float* s_q = s_k + W * DK;
  float* s_v = s_q + W * DK;
  float* s_b = s_v + W * NC;
  __shared__ float red_x[kWarps][NC];
  __shared__ float red_y[kWarps][NC];
  __shared__ float qk_part[2][kWarps];  // by token parity: the next token's partials may be
                                        // written while slower warps still read these
  __shared__ float tot_x[NC], tot_y[NC];

  const int slot = read_slots[b];
  if (slot < 0 || (int64_t)slot >= n_slots) {
    if ((int64_t)slot >= n_slots && threadIdx.x == 0 && h == 0 && part == 0 && status)
      atomicOr(status, KDA_STATUS_BAD_SLOT);
    for (int i = threadIdx.x; i < W * NC; i += blockDim.x) {
      const int j = i / NC, c = i - j * NC;
      st_elem(o, ((int64_t)(b * W + j) * H + h) * DV + part * NC + c, 0.0f);
    }
    return;
  }

  // Issue every state load of this thread first (RPW independent vector loads).
  const float* S = pool + ((int64_t)slot * H + h) * (int64_t)DK * DV;
  float st[RPW][CPL];
#pragma unroll
  for (int i = 0; i < RPW; ++i) {
    float2 t2 = __ldcs(reinterpret_cast<const float2*>(S + (int64_t)(r0 + i) * DV + cg));
    st[i][0] = t2.x; st[i][1] = t2.y;
  }

  // Stage the window's inputs (token-major rows: token b*W + j, head h).
  for (int i = threadIdx.x; i < W * DK; i += blockDim.x) {
    const int j = i / DK, c = i - j * DK;
    const int64_t e = ((int64_t)(b * W + j) * H + h) * DK + c;
    s_a[i] = __expf(g[e]);
    s_k[i] = ld_elem(k, e);
    s_q[i] = ld_elem(q, e);
  }
  for (int i = threadIdx.x; i < W * NC; i += blockDim.x) {
    const int j = i / NC, c = i - j * NC;
    s_v[i] = ld_elem(v, ((int64_t)(b * W + j) * H + h) * DV + part * NC + c);
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
    // decay in registers, then partial column sums over this warp's rows
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
    // column totals over the warps: one thread per (column, x|y)
    if (threadIdx.x < 2 * NC) {
      const int col = threadIdx.x % NC;
      float s = 0.0f;
      if (threadIdx.x < NC) {
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
      u[c] = s_v[j * NC + c0 + c] - x;
      if (warp == 0) st_elem(o, tok * DV + cg + c, scale * (y + bt * qk_all * u[c]));
    }
    // S' = Diag(a) S + beta k u^T
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
      const float bk = bt * kr[i];
#pragma unroll
      for (int c = 0; c < CPL; ++c) st[i][c] = fmaf(bk, u[c], st[i][c]);
    }

    // this column's snapshot
    const int ws = write_slots[(int64_t)b * W + j];
    if ((int64_t)ws >= n_slots) {
      if (threadIdx.x == 0 && h == 0 && part == 0 && status)
        atomicOr(status, KDA_STATUS_BAD_SLOT);
    } else if (ws >= 0) {
      float* D = pool + ((int64_t)ws * H + h) * (int64_t)DK * DV;
#pragma unroll
      for (int i = 0; i < RPW; ++i)
        __stcs(reinterpret_cast<float2*>(D + (int64_t)(r0 + i) * DV + cg),
               make_float2(st[i][0], st[i][1]));
    }
  }
}

template <int DK, int DV, class T>
kda_status launch_t(const char* fn, int batch, int window, int H, float scale, const void* q,
                    const void* k, const void* v, const float* g, const float* beta,
                    unsigned flags, const int32_t* read_slots, const int32_t* write_slots,
                    float* pool, int64_t n_slots, void* o, uint32_t* status, cudaStream_t s) {
  constexpr int NC = DV < kCols ? DV : kCols;
  const size_t smem = (size_t)window * (3 * DK + NC + 1) * sizeof(float);
  dim3 grid((unsigned)batch * (unsigned)H * (unsigned)(DV / NC));
  decode_kernel<DK, DV, T><<<grid, kWarps * 32, smem, s>>>(
      (const T*)q, (const T*)k, (const T*)v, g, beta, flags, read_slots, write_slots, pool,
      n_slots, H, window, scale, (T*)o, status);
  count_launches(1);
  return check_launch(fn);
}

kda_status dispatch(const char* fn, kda_dtype dt, int batch, int window, int H, int dk, int dv,
                    float scale, const void* q, const void* k, const void* v, const float* g,
                    const float* beta, unsigned flags, const int32_t* read_slots,
                    const int32_t* write_slots, float* pool, int64_t n_slots, void* o,
                    uint32_t* status, cudaStream_t s) {
  if (batch == 0 || window == 0) return KDA_OK;
  if (dk == 128 && dv == 128) {
    if (dt == KDA_BF16)
      return launch_t<128, 128, __nv_bfloat16>(fn, batch, window, H, scale, q, k, v, g, beta,
                                               flags, read_slots, write_slots, pool, n_slots, o,
                                               status, s);
    return launch_t<128, 128, float>(fn, batch, window, H, scale, q, k, v, g, beta, flags,
                                     read_slots, write_slots, pool, n_slots, o, status, s);
  }
  if (dk == 64 && dv == 64) {
    if (dt == KDA_BF16)
      return launch_t<64, 64, __nv_bfloat16>(fn, batch, window, H, scale, q, k, v, g, beta,
                                             flags, read_slots, write_slots, pool, n_slots, o,
                                             status, s);
    return launch_t<64, 64, float>(fn, batch, window, H, scale, q, k, v, g, beta, flags,
                                   read_slots, write_slots, pool, n_slots, o, status, s);
  }
  return set_error(KDA_ERR_UNSUPPORTED, std::string(fn) + ": dk = dv must be 64 or 128");
}

}  // namespace

kda_status launch_decode(kda_dtype dt, int batch, int H, int dk, int dv, float scale,
                         const void* q, const void* k, const void* v, const float* g,
                         const float* beta, const int32_t* slot_ids, float* pool,
                         int64_t n_slots, void* o, uint32_t* status, cudaStream_t s) {
  // one token per row, stored back into the slot it was read from
  return dispatch("kda_decode_step", dt, batch, 1, H, dk, dv, scale, q, k, v, g, beta, 0u,
                  slot_ids, slot_ids, pool, n_slots, o, status, s);
}

kda_status launch_decode_window(kda_dtype dt, int batch, int window, int H, int dk, int dv,
                                float scale, const void* q, const void* k, const void* v,
                                const float* g, const float* beta, unsigned flags,
                                const int32_t* read_slots, const int32_t* write_slots,
                                float* pool, int64_t n_slots, void* o, uint32_t* status,
                                cudaStream_t s) {
  return dispatch("kda_decode_window", dt, batch, window, H, dk, dv, scale, q, k, v, g, beta,
                  flags, read_slots, write_slots, pool, n_slots, o, status, s);
}

}  // namespace kda
