// Short causal depthwise convolution over packed varlen rows with a per-sequence history
// window in a slot pool: the KDA short-conv gather and window update.
//
// For sequence s and channel c, with history h = the W - 1 inputs before the sequence (oldest
// first, read from slot read_slots[s]; zeros for a negative id or no read table) and
// z = [h ; x_s]:
//     y_t = sum_{i=0}^{W-1} w[c, i] z[t - (W - 1) + i]      (w[c, W-1] weighs the current input)
//     out_t = y_t, or y_t / (1 + e^{-y_t}) with KDA_CONV_SILU,
// and the last W - 1 entries of z become the window stored into slot write_slots[s].
// Sources: kern PR #44 ("Prefill-only pipeline parallelism, from kern cut to full Kimi-K3"),
// squash message: the short-conv gather and window update are among the per-sequence kernels
// the stage split generalises to varlen rows (cu_seqlens); ATOM PR #2709 ("feat(kimi-k3): PP8
// prefill for P/D serving - KDA state under PP"): the speculative conv update reads its
// history through a read-side index. The pages give neither the width nor an activation, so
// both are arguments.
//
// HBM-bound stencil (W <= 4 multiply-adds per element). A CTA owns one tile of R tokens of
// one sequence (R = 32 for bf16, 16 for fp32) and 512 channels. One thread first brings the
// tile's rows and its W - 1 halo rows into shared memory with bulk tensor copies (boxes of
// [W - 1 + R rows][512 B] over the packed rows, completion on an mbarrier, bounded wait;
// ~35 KiB per CTA, so ~6 CTAs per SM have their copies in flight), then each thread computes
// 4 consecutive channels of every row from shared memory and stores them with streaming
// stores (a warp writes 32 x 4 contiguous elements per row). With bf16 the SiLU costs one
// special-function operation per element (see act()). The halo rows are the sequence's
// preceding inputs (read again, from L2) or, for its first tile, the history slot. The CTAs
// run channel block by channel block along a row tile. Tiles are placed like the chunk
// kernels' items: tile j of sequence s sits in slot floor(cu[s] / R) + s + j, and a CTA finds its
// sequence by binary search, so no host pass over the offsets is needed. Only the first tile
// of a sequence touches the history slots: the old window is in shared memory before it stores
// the new one, so read slot = write slot is safe.
#include "kda_internal.cuh"
#include "ptx.cuh"

namespace kda {
namespace {

constexpr int kThreads = 128;
constexpr int kBoxBytes = 512;            // inner extent of one bulk tensor copy
constexpr int kVec = 4;                   // channels per thread
constexpr int kCols = kThreads * kVec;    // channels per CTA

template <class T> constexpr int tile_rows() { return sizeof(T) == 2 ? 32 : 16; }

__device__ __forceinline__ float4 load4(const float* p) {
  return *reinterpret_cast<const float4*>(p);
}
__device__ __forceinline__ float4 load4(const __nv_bfloat16* p) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  __nv_bfloat162 a, b;
  memcpy(&a, &u.x, 4);
  memcpy(&b, &u.y, 4);
  const float2 fa = __bfloat1622float2(a), fb = __bfloat1622float2(b);
  return make_float4(fa.x, fa.y, fb.x, fb.y);
}
__device__ __forceinline__ void store4_smem(float* p, float4 v) {
  *reinterpret_cast<float4*>(p) = v;
}
__device__ __forceinline__ void store4_smem(__nv_bfloat16* p, float4 v) {
  const __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
  uint2 u;
  memcpy(&u.x, &a, 4);
  memcpy(&u.y, &b, 4);
  *reinterpret_cast<uint2*>(p) = u;
}
__device__ __forceinline__ void store4(float* p, float4 v) {
  __stcs(reinterpret_cast<float4*>(p), v);
}
__device__ __forceinline__ void store4(__nv_bfloat16* p, float4 v) {
  const __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
  uint2 u;
  memcpy(&u.x, &a, 4);
  memcpy(&u.y, &b, 4);
  __stcs(reinterpret_cast<uint2*>(p), u);
}
__device__ __forceinline__ float tanh_approx(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// SiLU y sigmoid(y). bf16 outputs: sigmoid(y) = (1 + tanh(y / 2)) / 2 with the hardware tanh,
// one special-function operation per element (relative error about 2^-11, far below the
// output's bf16 rounding). fp32 outputs: the fast exponential and division intrinsics (a few
// ulp; e^{-y} = inf for very negative y gives y * 0 = 0, the limit).
template <class T>
__device__ __forceinline__ float act(float y, bool silu) {
  if (!silu) return y;
  if (sizeof(T) == 2) {
    const float h = 0.5f * y;
    return fmaf(h, tanh_approx(h), h);
  }
  return __fdividef(y, 1.0f + __expf(-y));
}

template <int W, class T>
__global__ void __launch_bounds__(kThreads)
conv_kernel(const __grid_constant__ CUtensorMap xmap, const T* __restrict__ x,
            const float* __restrict__ w,
            const int32_t* __restrict__ cu, int n_seqs, int total, int C, unsigned flags,
            const int32_t* __restrict__ read_slots, const int32_t* __restrict__ write_slots,
            T* __restrict__ hist, int64_t n_slots, T* __restrict__ out, uint32_t* status) {
  constexpr int HW = W - 1;
  constexpr int R = tile_rows<T>();
  constexpr int ROWS = HW + R;
  constexpr int BC = kBoxBytes / (int)sizeof(T);  // channels per box
  // the tile: kCols / BC boxes of [ROWS][BC], each box dense (the bulk copy's layout)
  __shared__ __align__(128) T tile[kCols / BC][ROWS][BC];
  __shared__ uint64_t bar;
  // one-dimensional grid, channel blocks fastest: the CTAs in flight together cover whole
  // rows (contiguous runs of memory) rather than one column block of many rows
  const int ncb = (C + kCols - 1) / kCols;
  const int cblk = (int)(blockIdx.x % (unsigned)ncb);
  const int slot = (int)(blockIdx.x / (unsigned)ncb);
  const int cb = cblk * kCols;
  const int ncols = C - cb < kCols ? C - cb : kCols;
  const bool lead = (cblk == 0 && threadIdx.x == 0);  // reports status bits once
  int s = 0;
  if (cu) {  // largest s with floor(cu[s] / R) + s <= slot
    int lo = 0, hi = n_seqs - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (cu[mid] / R + mid <= slot) lo = mid;
      else hi = mid - 1;
    }
    s = lo;
  }
  const int64_t t0 = cu ? cu[s] : 0, t1 = cu ? cu[s + 1] : total;
  if (t0 < 0 || t1 < t0 || t1 > total) {
    if (lead && status) atomicOr(status, KDA_STATUS_BAD_OFFSETS);
    return;
  }
  const int64_t j = (int64_t)slot - (cu ? t0 / R + s : 0);
  const int64_t start = t0 + j * R;
  if (j < 0 || (j > 0 && start >= t1)) return;
  const int nrows = (int)((start + R < t1 ? start + R : t1) - start);

  int rs = -1, ws = -1;
  if (j == 0) {
    rs = read_slots ? read_slots[s] : -1;
    ws = write_slots ? write_slots[s] : -1;
    if ((int64_t)rs >= n_slots || (int64_t)ws >= n_slots) {
      if (lead && status) atomicOr(status, KDA_STATUS_BAD_SLOT);
      if ((int64_t)rs >= n_slots) rs = -1;
      if ((int64_t)ws >= n_slots) ws = -1;
    }
  }

  // rows 0 .. HW-1: the halo (preceding inputs), HW ..: the tile's rows, as kCols / BC bulk
  // tensor copies issued by one thread (rows before the first token or past the last, and
  // channels past C, arrive as zeros). A sequence's first tile then replaces the halo rows
  // with its old window, each thread for its own channels, which are the only ones it reads.
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar, 1);
    ptx::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    ptx::mbar_arrive_expect_tx(&bar, (uint32_t)(kCols / BC) * ROWS * kBoxBytes);
#pragma unroll
    for (int b = 0; b < kCols / BC; ++b)
      ptx::tma_load_2d(&tile[b][0][0], &xmap, &bar, cb + b * BC, (int)(start - HW));
  }
  const int cl = threadIdx.x * kVec;
  const int c = cb + cl;
  T* my = &tile[cl / BC][0][cl % BC];  // this thread's 4 channels of row 0 (rows BC apart)
  bool ok = ptx::mbar_wait(&bar, 0);
  if (!ok) {  // the copies never landed: report, let them finish (bounded) and stop
    if (status) atomicOr(status, KDA_STATUS_TIMEOUT);
    ptx::mbar_wait(&bar, 0, 100000000ull);
    return;
  }
  if (cl >= ncols) return;
  if (j == 0) {
#pragma unroll
    for (int i = 0; i < HW; ++i) {
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (rs >= 0) v = load4(hist + ((int64_t)rs * HW + i) * C + c);
      store4_smem(my + i * BC, v);
    }
  }
  float wt[kVec][W];
#pragma unroll
  for (int e = 0; e < kVec; ++e)
#pragma unroll
    for (int i = 0; i < W; ++i) wt[e][i] = __ldg(w + (int64_t)(c + e) * W + i);
  const bool silu = (flags & KDA_CONV_SILU) != 0;
  float4 z[W];  // rows r .. r + W - 1 of the tile: a ring, one shared-memory load per row
#pragma unroll
  for (int i = 0; i < HW; ++i) z[i] = load4(my + i * BC);
  for (int r = 0; r < nrows; ++r) {
    z[HW] = load4(my + (r + HW) * BC);
    float acc[kVec] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int i = 0; i < W; ++i) {
      acc[0] = fmaf(wt[0][i], z[i].x, acc[0]);
      acc[1] = fmaf(wt[1][i], z[i].y, acc[1]);
      acc[2] = fmaf(wt[2][i], z[i].z, acc[2]);
      acc[3] = fmaf(wt[3][i], z[i].w, acc[3]);
    }
    store4(out + (start + r) * C + c, make_float4(act<T>(acc[0], silu), act<T>(acc[1], silu),
                                                  act<T>(acc[2], silu), act<T>(acc[3], silu)));
#pragma unroll
    for (int i = 0; i < HW; ++i) z[i] = z[i + 1];
  }

  // window update: the last W - 1 entries of z = [old window ; x_s], i.e. z[L + r]; the tile
  // holds z[0 .. HW + nrows), the rest is read from x
  if (j == 0 && HW > 0 && ws >= 0) {
    const int64_t L = t1 - t0;
#pragma unroll
    for (int r = 0; r < HW; ++r) {
      const int64_t zi = L + r;
      const float4 v = zi < HW + nrows ? load4(my + zi * BC) : load4(x + (t0 + zi - HW) * C + c);
      store4(hist + ((int64_t)ws * HW + r) * C + c, v);
    }
  }
}

template <int W, class T>
bool launch_w(int n_seqs, int total, const int32_t* cu, int C, const void* x, const float* w,
              unsigned flags, const int32_t* rs, const int32_t* ws, void* hist, int64_t n_slots,
              void* out, uint32_t* status, cudaStream_t s) {
  CUtensorMap xmap;
  if (!make_map_rows(&xmap, x, sizeof(T) == 4, (uint64_t)C, (uint64_t)total,
                     (uint32_t)(kBoxBytes / sizeof(T)), (uint32_t)(W - 1 + tile_rows<T>())))
    return false;
  const int64_t tiles = (int64_t)total / tile_rows<T>() + n_seqs;
  const dim3 grid((unsigned)(tiles * ((C + kCols - 1) / kCols)));
  conv_kernel<W, T><<<grid, kThreads, 0, s>>>(xmap, (const T*)x, w, cu, n_seqs, total, C, flags,
                                              rs, ws, (T*)hist, n_slots, (T*)out, status);
  return true;
}

template <class T>
bool launch_t(int width, int n_seqs, int total, const int32_t* cu, int C, const void* x,
              const float* w, unsigned flags, const int32_t* rs, const int32_t* ws, void* hist,
              int64_t n_slots, void* out, uint32_t* status, cudaStream_t s) {
  switch (width) {
    case 1: return launch_w<1, T>(n_seqs, total, cu, C, x, w, flags, rs, ws, hist, n_slots, out, status, s);
    case 2: return launch_w<2, T>(n_seqs, total, cu, C, x, w, flags, rs, ws, hist, n_slots, out, status, s);
    case 3: return launch_w<3, T>(n_seqs, total, cu, C, x, w, flags, rs, ws, hist, n_slots, out, status, s);
    default: return launch_w<4, T>(n_seqs, total, cu, C, x, w, flags, rs, ws, hist, n_slots, out, status, s);
  }
}

}  // namespace

kda_status launch_short_conv(kda_dtype dt, int n_seqs, int total, const int32_t* cu, int C,
                             int width, const void* x, const float* w, unsigned flags,
                             const int32_t* read_slots, const int32_t* write_slots, void* hist,
                             int64_t n_slots, void* out, uint32_t* status, cudaStream_t s) {
  if (n_seqs == 0) return KDA_OK;
  const bool ok =
      dt == KDA_BF16
          ? launch_t<__nv_bfloat16>(width, n_seqs, total, cu, C, x, w, flags, read_slots,
                                    write_slots, hist, n_slots, out, status, s)
          : launch_t<float>(width, n_seqs, total, cu, C, x, w, flags, read_slots, write_slots,
                            hist, n_slots, out, status, s);
  if (!ok)
    return set_error(KDA_ERR_UNSUPPORTED,
                     "kda_short_conv: cuTensorMapEncodeTiled is unavailable or rejected the "
                     "layout of x");
  count_launches(1);
  return check_launch("kda_short_conv");
}

}  // namespace kda
