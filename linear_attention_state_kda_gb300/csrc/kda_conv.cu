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
// HBM-bound stencil (W <= 4 multiply-adds per element). The work items are tiles of R tokens
// of one sequence (R = 32 for bf16, 16 for fp32) by 512 channels, channel blocks fastest, so
// that the items in flight together cover whole rows (contiguous runs of memory). A persistent
// grid of 3 CTAs per SM (a multiple of the channel-block count where it can be, so that a CTA
// keeps one block and its taps in registers) takes items b, b + G, b + 2G, ... through two
// shared-memory stages: one thread brings an item's rows and its W - 1 halo rows in with bulk
// tensor copies (boxes of [W - 1 + R rows][512 B] over the packed rows, completion on the
// stage's mbarrier, bounded wait; ~35 KiB a stage for bf16) and decodes the item (sequence,
// tile, rows) into the stage once, while the CTA computes the previous stage; each thread
// computes 4 consecutive channels of every row from shared memory and stores them with
// streaming stores (a warp writes 32 x 4 contiguous elements per row). With bf16 the SiLU
// costs one special-function operation per element (see act()). The halo rows are the
// sequence's preceding inputs (read again, from L2) or, for its first tile, the history slot.
// Tiles are placed like the chunk kernels' items: tile j of sequence s sits in slot
// floor(cu[s] / R) + s + j (a slot past a sequence's last tile is a hole), and the issuing
// thread finds an item's sequence by binary search, so no host pass over the offsets is
// needed. Only the first tile of a sequence touches the history slots: the old window is in
// shared memory before it stores the new one, so read slot = write slot is safe.
// Measured against the one-tile-per-CTA form (6 CTAs per SM, one copy each, every CTA decoding
// its own item): 0.1300 vs 0.1330 ms on 16k tokens x 12288 channels in a loop of itself and
// 0.131 vs 0.135 ms after a write-heavy kernel left L2 dirty. Fewer CTAs per SM with deeper
// stages, smaller tiles, or two thread groups splitting a tile's rows were all slower (fewer
// warps to cover each row's dependent arithmetic, or fewer bytes in flight).
#include "kda_internal.cuh"
#include "ptx.cuh"

namespace kda {
namespace {

constexpr int kThreads = 128;
constexpr int kBoxBytes = 512;            // inner extent of one bulk tensor copy
constexpr int kVec = 4;                   // channels per thread
constexpr int kCols = kThreads * kVec;    // channels per CTA
constexpr int kStages = 2;                // tile buffers per CTA
constexpr int kCtasPerSm = 3;             // persistent CTAs per SM

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

// Tile geometry of one pipeline stage: kCols / BC boxes of [ROWS][BC], each box dense (the bulk
// copy's layout); rows 0 .. HW-1 are the halo (the W - 1 inputs before the tile).
template <int W, class T>
struct TileShape {
  static constexpr int HW = W - 1;
  static constexpr int R = tile_rows<T>();
  static constexpr int ROWS = HW + R;
  static constexpr int BC = kBoxBytes / (int)sizeof(T);  // channels per box
  static constexpr int NB = kCols / BC;                  // boxes per tile
  static constexpr int ELEMS = NB * ROWS * BC;
  static constexpr uint32_t BYTES = (uint32_t)ELEMS * (uint32_t)sizeof(T);
};

// Work item `item` (channel blocks fastest, then tile slots): its sequence, tile and channel
// block. Tile j of sequence s sits in slot floor(cu[s] / R) + s + j; a slot past the sequence's
// last tile is a hole (valid = false); a sequence's first tile is valid even when it is empty,
// since it still carries the history window over.
struct ConvItem {
  int64_t t0, t1, start, j;
  int s, cb, ncols, nrows;
  bool valid, bad;
};

template <int R>
__device__ __forceinline__ ConvItem conv_item(int item, int ncb, const int32_t* __restrict__ cu,
                                              int n_seqs, int total, int C) {
  ConvItem it;
  it.valid = false;
  it.bad = false;
  it.nrows = 0;
  const int slot = item / ncb;
  it.cb = (item - slot * ncb) * kCols;
  it.ncols = C - it.cb < kCols ? C - it.cb : kCols;
  int s = 0;
  if (cu) {  // largest s with floor(cu[s] / R) + s <= slot
    int lo = 0, hi = n_seqs - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if ((int64_t)(cu[mid] / R) + mid <= slot) lo = mid;
      else hi = mid - 1;
    }
    s = lo;
  }
  it.s = s;
  it.t0 = cu ? cu[s] : 0;
  it.t1 = cu ? cu[s + 1] : total;
  if (it.t0 < 0 || it.t1 < it.t0 || it.t1 > total) {
    it.bad = true;
    return it;
  }
  it.j = slot - (cu ? it.t0 / R + s : 0);
  it.start = it.t0 + it.j * R;
  if (it.j < 0 || (it.j > 0 && it.start >= it.t1)) return it;
  it.nrows = (int)((it.start + R < it.t1 ? it.start + R : it.t1) - it.start);
  it.valid = true;
  return it;
}

// Persistent: CTA b takes items b, b + G, b + 2G, ... (G = gridDim.x) through kStages tile
// buffers. One thread keeps the copies of the next kStages - 1 items in flight while the CTA
// computes the current one, so every CTA always has tile bytes on the way from HBM.
template <int W, class T>
__global__ void __launch_bounds__(kThreads)
conv_kernel(const __grid_constant__ CUtensorMap xmap, const T* __restrict__ x,
            const float* __restrict__ w,
            const int32_t* __restrict__ cu, int n_seqs, int total, int C, unsigned flags,
            const int32_t* __restrict__ read_slots, const int32_t* __restrict__ write_slots,
            T* __restrict__ hist, int64_t n_slots, T* __restrict__ out, int n_items,
            uint32_t* status) {
  using S = TileShape<W, T>;
  constexpr int HW = S::HW, R = S::R, BC = S::BC;
  extern __shared__ uint8_t conv_smem[];  // rounded up to 128 B (bulk copy destinations)
  T* const tiles = reinterpret_cast<T*>(((uintptr_t)conv_smem + 127) & ~(uintptr_t)127);
  __shared__ uint64_t bar[kStages];
  __shared__ ConvItem info[kStages];  // the item in each stage, decoded once by the issuer
  const int ncb = (C + kCols - 1) / kCols;
  const int G = (int)gridDim.x;

  // rows 0 .. HW-1 of a stage: the halo, HW ..: the tile's rows, as NB bulk tensor copies
  // (rows before the first token or past the last, and channels past C, arrive as zeros); a
  // hole completes its stage's phase with a plain arrival, so that the phases stay in step
  auto issue = [&](int item, int st) {
    const ConvItem it = conv_item<R>(item, ncb, cu, n_seqs, total, C);
    if (it.bad && it.cb == 0 && status) atomicOr(status, KDA_STATUS_BAD_OFFSETS);
    info[st] = it;  // published by the arrival below (release) to the stage's waiters
    if (!it.valid) {
      ptx::mbar_arrive(&bar[st]);
      return;
    }
    ptx::mbar_arrive_expect_tx(&bar[st], S::BYTES);
    T* dst = tiles + st * S::ELEMS;
#pragma unroll
    for (int b = 0; b < S::NB; ++b)
      ptx::tma_load_2d(dst + b * S::ROWS * BC, &xmap, &bar[st], it.cb + b * BC,
                       (int)(it.start - HW));
  };
  if (threadIdx.x == 0) {
#pragma unroll
    for (int st = 0; st < kStages; ++st) ptx::mbar_init(&bar[st], 1);
    ptx::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
#pragma unroll
    for (int st = 0; st < kStages; ++st)
      if (blockIdx.x + st * G < n_items) issue(blockIdx.x + st * G, st);
  }

  const int cl = threadIdx.x * kVec;
  const int off = (cl / BC) * S::ROWS * BC + cl % BC;  // this thread's 4 channels of row 0
  const bool silu = (flags & KDA_CONV_SILU) != 0;
  float wt[kVec][W];  // the taps of this thread's channels, loaded when the block changes
  int wcb = -1;
  int k = 0;
  for (int item = blockIdx.x; item < n_items; item += G, ++k) {
    const int st = k % kStages;
    const bool landed = ptx::mbar_wait(&bar[st], (uint32_t)(k / kStages) & 1u);
    const ConvItem it = info[st];
    const int c = it.cb + cl;
    if (landed && it.valid && cl < it.ncols) {
      T* my = tiles + st * S::ELEMS + off;  // rows BC apart
      int rs = -1, ws = -1;
      if (it.j == 0) {
        rs = read_slots ? read_slots[it.s] : -1;
        ws = write_slots ? write_slots[it.s] : -1;
        if ((int64_t)rs >= n_slots || (int64_t)ws >= n_slots) {
          if (it.cb == 0 && threadIdx.x == 0 && status) atomicOr(status, KDA_STATUS_BAD_SLOT);
          if ((int64_t)rs >= n_slots) rs = -1;
          if ((int64_t)ws >= n_slots) ws = -1;
        }
        // a sequence's first tile: its halo rows are the old window, each thread writing its
        // own channels, the only ones it reads
#pragma unroll
        for (int i = 0; i < HW; ++i) {
          float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
          if (rs >= 0) v = load4(hist + ((int64_t)rs * HW + i) * C + c);
          store4_smem(my + i * BC, v);
        }
      }
      if (it.cb != wcb) {
        wcb = it.cb;
#pragma unroll
        for (int e = 0; e < kVec; ++e)
#pragma unroll
          for (int i = 0; i < W; ++i) wt[e][i] = __ldg(w + (int64_t)(c + e) * W + i);
      }
      float4 z[W];  // rows r .. r + W - 1 of the tile: a ring, one shared-memory load per row
#pragma unroll
      for (int i = 0; i < HW; ++i) z[i] = load4(my + i * BC);
      T* dst = out + it.start * C + c;
      for (int r = 0; r < it.nrows; ++r) {
        z[HW] = load4(my + (r + HW) * BC);
        float acc[kVec] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int i = 0; i < W; ++i) {
          acc[0] = fmaf(wt[0][i], z[i].x, acc[0]);
          acc[1] = fmaf(wt[1][i], z[i].y, acc[1]);
          acc[2] = fmaf(wt[2][i], z[i].z, acc[2]);
          acc[3] = fmaf(wt[3][i], z[i].w, acc[3]);
        }
        store4(dst + (int64_t)r * C, make_float4(act<T>(acc[0], silu), act<T>(acc[1], silu),
                                                 act<T>(acc[2], silu), act<T>(acc[3], silu)));
#pragma unroll
        for (int i = 0; i < HW; ++i) z[i] = z[i + 1];
      }
      // window update: the last W - 1 entries of z = [old window ; x_s], i.e. z[L + r]; the
      // tile holds z[0 .. HW + nrows), the rest is read from x
      if (it.j == 0 && HW > 0 && ws >= 0) {
        const int64_t L = it.t1 - it.t0;
#pragma unroll
        for (int r = 0; r < HW; ++r) {
          const int64_t zi = L + r;
          const float4 v = zi < HW + it.nrows ? load4(my + zi * BC)
                                              : load4(x + (it.t0 + zi - HW) * C + c);
          store4(hist + ((int64_t)ws * HW + r) * C + c, v);
        }
      }
    }
    // every thread is done with the stage (its generic-proxy reads and halo writes ordered
    // before the next bulk copy into it); then refill it with item k + kStages
    ptx::fence_proxy_async_smem();
    if (__syncthreads_or(!landed)) {
      // a copy never landed: report, let this CTA's copies in flight finish (bounded), stop
      if (threadIdx.x == 0) {
        if (status) atomicOr(status, KDA_STATUS_TIMEOUT);
        for (int i = 0; i < kStages; ++i) {
          const int kk = k + i;
          if (blockIdx.x + kk * G < n_items)
            ptx::mbar_wait(&bar[kk % kStages], (uint32_t)(kk / kStages) & 1u, 100000000ull);
        }
      }
      return;
    }
    if (threadIdx.x == 0 && item + kStages * G < n_items) issue(item + kStages * G, st);
  }
}

int conv_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    n = 148;
  return n;
}

template <int W, class T>
bool launch_w(int n_seqs, int total, const int32_t* cu, int C, const void* x, const float* w,
              unsigned flags, const int32_t* rs, const int32_t* ws, void* hist, int64_t n_slots,
              void* out, uint32_t* status, cudaStream_t s) {
  using S = TileShape<W, T>;
  CUtensorMap xmap;
  if (!make_map_rows(&xmap, x, sizeof(T) == 4, (uint64_t)C, (uint64_t)total, (uint32_t)S::BC,
                     (uint32_t)S::ROWS))
    return false;
  constexpr size_t smem = (size_t)kStages * S::BYTES + 128;
  // CTAs resident per SM at this shared-memory size (at most kCtasPerSm), so that every CTA
  // of the persistent grid runs from the start; the attribute and the query are per device,
  // done on a device's first call (a repeated first call just does them again)
  static int per_sm_of[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return false;
  int per_sm = dev < 64 ? per_sm_of[dev] : 0;
  if (per_sm <= 0) {
    int n = 0;
    if (cudaFuncSetAttribute(conv_kernel<W, T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, conv_kernel<W, T>, kThreads, smem) !=
            cudaSuccess)
      return false;
    per_sm = n < kCtasPerSm ? n : kCtasPerSm;
    if (dev < 64) per_sm_of[dev] = per_sm;
  }
  if (per_sm <= 0) return false;
  const int64_t tiles = (int64_t)total / S::R + n_seqs;
  const int64_t ncb = (C + kCols - 1) / kCols;
  const int64_t n_items = tiles * ncb;
  if (n_items > INT32_MAX / 2) return false;
  // a multiple of the channel-block count when it can be: each CTA then keeps one block (and
  // its taps in registers) throughout
  const int64_t cap = (int64_t)conv_sm_count() * per_sm;
  const int64_t full = cap >= ncb ? cap / ncb * ncb : cap;
  const unsigned grid = (unsigned)(n_items < full ? n_items : full);
  conv_kernel<W, T><<<grid, kThreads, smem, s>>>(xmap, (const T*)x, w, cu, n_seqs, total, C,
                                                 flags, rs, ws, (T*)hist, n_slots, (T*)out,
                                                 (int)n_items, status);
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
                     "layout of x, the kernel's shared memory could not be reserved, or x has "
                     "more than 2^30 tiles");
  count_launches(1);
  return check_launch("kda_short_conv");
}

}  // namespace kda
