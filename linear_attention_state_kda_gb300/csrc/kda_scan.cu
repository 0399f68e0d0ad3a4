// Segmented exclusive prefix over KDA segment packages.
//
// A package (M, D) maps a segment's entry state to its exit state, S_out = M S_in + D, and
// two consecutive packages combine as (M2, D2) o (M1, D1) = (M2 M1, M2 D1 + D2) ("apply 1,
// then 2"). pegainfer PR #970 (whale-rendezvous and fabric data-plane commit messages)
// exchanges these KDA (M,D) packages between context-parallel ranks and names a Blelloch
// prefix scan as the lower-traffic way to combine them. On one GPU this file offers two
// schedules of the same prefix (equal up to rounding order), per (sequence, head):
//   * the sequential chain (namespace seqtc, dk = dv = 128, up to 256 segments per sequence):
//     S_0 = S_init, seg_init[j] = S_j, S_{j+1} = M_j S_j + D_j, one dependent tensor-core
//     product per segment, the state's columns split over CTAs;
//   * the work-efficient (Blelloch) tree, for longer sequences and for dk = dv = 64:
//       - the sequence's packages are copied into a power-of-two tree, padded with (I, 0);
//       - up-sweep: at stride d, node i (i+1 multiple of 2d) becomes a[i] o a[i-d];
//       - the root (the whole sequence's package) gives the exit state, then becomes (I, 0);
//       - down-sweep: at stride d, (a[i-d], a[i]) <- (a[i], a[i-d] o a[i]);
//       - leaf j then holds the exclusive prefix (M_<j, D_<j), and the segment's entry state
//         is M_<j S_init + D_<j.
//     Every combine is a dk x dk times dk x (dk + dv) product. For dk = dv = 128 the whole
//     tree of a (sequence, head) runs in one launch, one cluster of 4 CTAs per tree, every
//     combine and entry-state application on tcgen05 tensor cores with a 3xTF32 split
//     (namespace tc). The CUDA-core version (dk = 64) has a CTA compute a 32-row block of one
//     combine's result: it reads only its own rows of the left operand, so that storage can
//     take the result in place.
#include "kda_internal.cuh"
#include "ptx.cuh"

namespace kda {
namespace {

constexpr int kRows = 32;       // rows of the result per CTA
constexpr int kThreads = 256;

__host__ __device__ inline int64_t pkg_floats(int dk, int dv) {
  return (int64_t)dk * dk + (int64_t)dk * dv;
}

struct Tree {
  float* base;    // [n_seqs][P2][H] packages (M then D)
  float* tmp;     // [n_seqs][P2/2][H] packages
  int P2, H, dk, dv, n_segs, max_segs;
  // Segment range of sequence s, or an empty range if the offsets are malformed.
  __device__ bool seq_range(const int32_t* off, int s, int& first, int& cnt) const {
    first = off[s];
    cnt = off[s + 1] - first;
    if (first < 0 || cnt < 0 || cnt > max_segs || first + cnt > n_segs) {
      first = 0;
      cnt = 0;
      return false;
    }
    return true;
  }
  __device__ float* node(int s, int i, int h) const {
    return base + (((int64_t)s * P2 + i) * H + h) * pkg_floats(dk, dv);
  }
  __device__ float* tnode(int s, int i, int h) const {
    return tmp + (((int64_t)s * (P2 / 2) + i) * H + h) * pkg_floats(dk, dv);
  }
};

// Copy each sequence's packages into its padded tree; pad with (I, 0).
__global__ void scan_fill(Tree t, const float* __restrict__ M, const float* __restrict__ D,
                          const int32_t* __restrict__ seq_off, uint32_t* status) {
  const int i = blockIdx.x, h = blockIdx.y, s = blockIdx.z;
  int first, cnt;
  if (!t.seq_range(seq_off, s, first, cnt) && i == 0 && h == 0 && threadIdx.x == 0 && status)
    atomicOr(status, KDA_STATUS_BAD_OFFSETS);
  float* dst = t.node(s, i, h);
  const int dk = t.dk, dv = t.dv;
  if (i < cnt) {
    const float* m = M + ((int64_t)(first + i) * t.H + h) * dk * dk;
    const float* d = D + ((int64_t)(first + i) * t.H + h) * dk * dv;
    for (int e = threadIdx.x; e < dk * dk; e += blockDim.x) dst[e] = m[e];
    for (int e = threadIdx.x; e < dk * dv; e += blockDim.x) dst[dk * dk + e] = d[e];
  } else {
    for (int e = threadIdx.x; e < dk * dk; e += blockDim.x)
      dst[e] = (e / dk == e % dk) ? 1.0f : 0.0f;
    for (int e = threadIdx.x; e < dk * dv; e += blockDim.x) dst[dk * dk + e] = 0.0f;
  }
}

// out = A o B for rows [r0, r0 + 32): out.M = A.M B.M, out.D = A.M B.D + A.D.
// out may be A's storage (each CTA reads its rows of A before writing them).
template <int DK, int DV>
__device__ void combine_rows(const float* A, const float* B, float* out, int r0) {
  __shared__ float Am[kRows][DK + 1];
  __shared__ float Ad[kRows][DV];
  for (int e = threadIdx.x; e < kRows * DK; e += blockDim.x)
    Am[e / DK][e % DK] = A[(int64_t)(r0 + e / DK) * DK + e % DK];
  for (int e = threadIdx.x; e < kRows * DV; e += blockDim.x)
    Ad[e / DV][e % DV] = A[DK * DK + (int64_t)(r0 + e / DV) * DV + e % DV];
  __syncthreads();
  constexpr int W = DK + DV;  // result columns
  for (int col = threadIdx.x; col < W; col += blockDim.x) {
    const float* bcol = col < DK ? B + col : B + DK * DK + (col - DK);
    const int ld = col < DK ? DK : DV;
    float acc[kRows];
#pragma unroll
    for (int r = 0; r < kRows; ++r) acc[r] = col < DK ? 0.0f : Ad[r][col - DK];
    for (int x = 0; x < DK; ++x) {
      const float b = bcol[(int64_t)x * ld];
#pragma unroll
      for (int r = 0; r < kRows; ++r) acc[r] = fmaf(Am[r][x], b, acc[r]);
    }
    float* dst = col < DK ? out + col : out + DK * DK + (col - DK);
#pragma unroll
    for (int r = 0; r < kRows; ++r) dst[(int64_t)(r0 + r) * ld] = acc[r];
  }
}

// Up-sweep level d: node i = (2*pair + 2)*d - 1 becomes a[i] o a[i-d].
template <int DK, int DV>
__global__ void __launch_bounds__(kThreads) scan_up(Tree t, int d) {
  const int pair = blockIdx.x, h = blockIdx.y / (DK / kRows);
  const int r0 = (blockIdx.y % (DK / kRows)) * kRows, s = blockIdx.z;
  const int i = (2 * pair + 2) * d - 1;
  combine_rows<DK, DV>(t.node(s, i, h), t.node(s, i - d, h), t.node(s, i, h), r0);
}

// Down-sweep level d, first half: tmp[pair] = a[i-d] o a[i].
template <int DK, int DV>
__global__ void __launch_bounds__(kThreads) scan_down_combine(Tree t, int d) {
  const int pair = blockIdx.x, h = blockIdx.y / (DK / kRows);
  const int r0 = (blockIdx.y % (DK / kRows)) * kRows, s = blockIdx.z;
  const int i = (2 * pair + 2) * d - 1;
  combine_rows<DK, DV>(t.node(s, i - d, h), t.node(s, i, h), t.tnode(s, pair, h), r0);
}

// Down-sweep level d, second half: a[i-d] <- a[i]; a[i] <- tmp[pair].
__global__ void scan_down_move(Tree t, int d) {
  const int pair = blockIdx.x, h = blockIdx.y, s = blockIdx.z;
  const int i = (2 * pair + 2) * d - 1;
  const int64_t n = pkg_floats(t.dk, t.dv);
  float* L = t.node(s, i - d, h);
  float* R = t.node(s, i, h);
  const float* X = t.tnode(s, pair, h);
  for (int64_t e = threadIdx.x; e < n; e += blockDim.x) {
    L[e] = R[e];
    R[e] = X[e];
  }
}

// Applies package P (M then D) to S_init rows [r0, r0+32): out = M S_init + D (D if no init).
template <int DK, int DV>
__device__ void apply_rows(const float* P, const float* S_init, float* out, int r0) {
  __shared__ float Am[kRows][DK + 1];
  for (int e = threadIdx.x; e < kRows * DK; e += blockDim.x)
    Am[e / DK][e % DK] = P[(int64_t)(r0 + e / DK) * DK + e % DK];
  __syncthreads();
  for (int col = threadIdx.x; col < DV; col += blockDim.x) {
    for (int r = 0; r < kRows; ++r) {
      float acc = P[DK * DK + (int64_t)(r0 + r) * DV + col];
      if (S_init)
        for (int x = 0; x < DK; ++x) acc = fmaf(Am[r][x], S_init[(int64_t)x * DV + col], acc);
      out[(int64_t)(r0 + r) * DV + col] = acc;
    }
  }
}

// Root: exit state from the whole-sequence package, then reset the root to (I, 0).
template <int DK, int DV>
__global__ void __launch_bounds__(kThreads) scan_root(Tree t, const float* init,
                                                      float* final_state) {
  const int h = blockIdx.y / (DK / kRows);
  const int r0 = (blockIdx.y % (DK / kRows)) * kRows, s = blockIdx.z;
  float* root = t.node(s, t.P2 - 1, h);
  const int64_t sd = (int64_t)DK * DV;
  const float* si = init ? init + ((int64_t)s * t.H + h) * sd : nullptr;
  if (final_state) apply_rows<DK, DV>(root, si, final_state + ((int64_t)s * t.H + h) * sd, r0);
  __syncthreads();
  for (int e = threadIdx.x; e < kRows * DK; e += blockDim.x) {
    const int r = r0 + e / DK, c = e % DK;
    root[(int64_t)r * DK + c] = (r == c) ? 1.0f : 0.0f;
  }
  for (int e = threadIdx.x; e < kRows * DV; e += blockDim.x)
    root[DK * DK + (int64_t)(r0 + e / DV) * DV + e % DV] = 0.0f;
}

// Entry state of segment j of sequence s from its exclusive prefix.
template <int DK, int DV>
__global__ void __launch_bounds__(kThreads) scan_apply(Tree t, const int32_t* seq_off,
                                                       const float* init, float* seg_init) {
  const int j = blockIdx.x, h = blockIdx.y / (DK / kRows);
  const int r0 = (blockIdx.y % (DK / kRows)) * kRows, s = blockIdx.z;
  int first, cnt;
  t.seq_range(seq_off, s, first, cnt);
  if (j >= cnt) return;
  const int64_t sd = (int64_t)DK * DV;
  const float* si = init ? init + ((int64_t)s * t.H + h) * sd : nullptr;
  apply_rows<DK, DV>(t.node(s, j, h), si, seg_init + ((int64_t)(first + j) * t.H + h) * sd, r0);
}

// ------------------------------------------------------------------ tensor-core combines
// For dk = dv = 128 the combines run on tcgen05: a CTA computes one 64-column tile of
// out = A o B = (A.M B.M, A.M B.D + A.D) (or of a prefix applied to an entry state,
// out.D = A.M S + A.D). A.M is the K-major A operand (128 x 128); the tile of [B.M | B.D] is
// staged transposed as the K-major B operand (64 x 128); the product accumulates in TMEM.
// Every product is split 3xTF32 to keep fp32-level accuracy through the tree's levels:
//   X = X_hi + X_lo, X_hi = X with its low 13 mantissa bits cleared (what a tf32 MMA reads),
//   X_lo = X - X_hi (exact); A B ~ A_hi B_hi + A_hi B_lo + A_lo B_hi  (error ~ 2^-21 rel.).
// A combine's result goes to a separate node (tmp) because every tile CTA reads all of A.
namespace tc {

using namespace ptx;

constexpr int DK = 128;
constexpr int NT = 64;                          // output columns per CTA
constexpr uint32_t A_KB = 128 * 128;            // A operand K-block: 128 rows x 128 B
constexpr uint32_t B_KB = NT * 128;             // B operand K-block: 64 rows x 128 B
constexpr uint32_t AH = 0, AL = 4 * A_KB, BH = 8 * A_KB, BL = 8 * A_KB + 4 * B_KB;
constexpr uint32_t SMEM = BL + 4 * B_KB + 1024;  // + alignment slack

__device__ __forceinline__ float hi(float x) {
  return __uint_as_float(__float_as_uint(x) & 0xFFFFE000u);
}

// ------------------------------------------------------------ whole tree in one launch
// One cluster of 4 CTAs per (sequence, head) runs fill, up-sweep, root, down-sweep and the
// entry-state applications; CTA r owns column tile r of every combine (tiles 0, 1: M columns,
// 2, 3: D columns). Every combine reads the whole left operand, so a level writes its results
// to the tmp nodes, and after a cluster barrier each CTA moves its own tiles into place.
// TMEM (64 columns) and the operand barrier live for the whole kernel.

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

struct TileCtx {
  uint32_t tbase;
  uint64_t* bar;
  uint32_t phase;
  bool ok;
};

// A.M (row-major 128 x 128) -> the A operand in shared memory, split 3xTF32 (hi / lo, K-major).
// Every load is issued before the first shared-memory store (one round trip to L2).
__device__ void load_a(const float* A) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const int tid = threadIdx.x;
  float4 a[16];
#pragma unroll
  for (int u = 0; u < 16; ++u) {  // element e = tid + 256 u
    const int e = tid + u * kThreads;
    a[u] = *reinterpret_cast<const float4*>(A + (e >> 5) * DK + (e & 31) * 4);
  }
#pragma unroll
  for (int u = 0; u < 16; ++u) {
    const int e = tid + u * kThreads;
    const float4 hh = make_float4(hi(a[u].x), hi(a[u].y), hi(a[u].z), hi(a[u].w));
    const uint32_t off = sw128_off32(e >> 5, (e & 31) * 4, A_KB);
    *reinterpret_cast<float4*>(sm + AH + off) = hh;
    *reinterpret_cast<float4*>(sm + AL + off) =
        make_float4(a[u].x - hh.x, a[u].y - hh.y, a[u].z - hh.z, a[u].w - hh.w);
  }
}

// One 64-column tile of out = A o B with A.M already in shared memory (load_a, then a barrier
// that orders it before the product): tiles 0, 1 are out.M = A.M B.M, tiles 2, 3 out.D =
// A.M B.D + A.D (bm null: a state application, out.D = A.M S + A.D with S = bd; bd null as well:
// out.D = A.D). ad is A.D. TMEM and the barrier come with the context.
__device__ void tile_product(TileCtx& cx, const float* ad_pkg, const float* bm, const float* bd,
                             float* om, float* od, int tile, uint32_t* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool mtile = tile < DK / NT;
  const int col0 = (mtile ? tile : tile - DK / NT) * NT;
  float* out = mtile ? om : od;
  const float* B = mtile ? bm : bd;
  // A.D's part of this tile (D tiles), loaded now so that its latency hides under the product
  float4 adv[8];
  const int r = (warp & 3) * 32 + lane, cb = (warp >> 2) * 32;
  if (!mtile) {
    const float4* ad = reinterpret_cast<const float4*>(ad_pkg + r * DK + col0 + cb);
#pragma unroll
    for (int j = 0; j < 8; ++j) adv[j] = ad[j];
  }
  if (B) {
    // the B tile: element e = tid + 256 u is row k = (e & 127) of columns n4 .. n4 + 3,
    // n4 = 4 (e >> 7), so that a warp's transposed stores below fill whole 128-byte rows
    float4 b[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int e = tid + u * kThreads;
      b[u] = *reinterpret_cast<const float4*>(B + (e & 127) * DK + col0 + (e >> 7) * 4);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {  // B tile, transposed (row n, 32 consecutive k per warp)
      const int e = tid + u * kThreads;
      const int k = e & 127, n4 = (e >> 7) * 4;
      const float bv[4] = {b[u].x, b[u].y, b[u].z, b[u].w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t off = sw128_off32(n4 + q, k, B_KB);
        const float h = hi(bv[q]);
        *reinterpret_cast<float*>(sm + BH + off) = h;
        *reinterpret_cast<float*>(sm + BL + off) = bv[q] - h;
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) {
      const uint32_t sb = smem_u32(sm);
      const uint32_t idesc = idesc_make(kFmtTF32, 128, NT, false, false);
      const uint64_t dah = sdesc_sw128(sb + AH, 16, 1024), dal = sdesc_sw128(sb + AL, 16, 1024);
      const uint64_t dbh = sdesc_sw128(sb + BH, 16, 1024), dbl = sdesc_sw128(sb + BL, 16, 1024);
#pragma unroll
      for (int s = 0; s < 16; ++s) {
        const uint32_t ka = (s >> 2) * A_KB + (s & 3) * 32, kb = (s >> 2) * B_KB + (s & 3) * 32;
        const uint64_t ah = desc_add(dah, ka), al = desc_add(dal, ka);
        const uint64_t bh = desc_add(dbh, kb), bl = desc_add(dbl, kb);
        mma_tf32(cx.tbase, ah, bh, idesc, s > 0 ? 1u : 0u);
        mma_tf32(cx.tbase, ah, bl, idesc, 1);
        mma_tf32(cx.tbase, al, bh, idesc, 1);
      }
      mma_commit(cx.bar);
    }
    const bool ok = mbar_wait(cx.bar, cx.phase);
    cx.phase ^= 1u;
    if (!ok) {
      cx.ok = false;
      if (tid == 0 && status) atomicOr(status, KDA_STATUS_TIMEOUT);
    }
    tc_fence_after();
  }
  {  // warp w: rows 32 (w % 4).., columns 32 (w / 4)..; D tiles add A.D
    float v[32];
    if (B) {
      tmem_ld32(cx.tbase + ((uint32_t)((warp & 3) * 32) << 16) + cb, v);
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = 0.0f;
    }
    if (!mtile) {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        v[4 * j] += adv[j].x; v[4 * j + 1] += adv[j].y; v[4 * j + 2] += adv[j].z;
        v[4 * j + 3] += adv[j].w;
      }
    }
    float* dst = out + r * DK + col0 + cb;
#pragma unroll
    for (int j = 0; j < 32; j += 4)
      *reinterpret_cast<float4*>(dst + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
  }
  tc_fence_before();
  __syncthreads();  // the B buffers and TMEM are reused by the next tile
  tc_fence_after();
}

// Work of one tree level with `pairs` combines, over the cluster's 4 CTAs: with 4 or more
// combines a CTA takes whole combines (its A operand loaded once for all 4 tiles); with 2, two
// CTAs share a combine (2 tiles each); with 1, each CTA takes one tile. Returns the tiles of
// round `round` for this CTA: combine index `pair`, tiles [t0, t0 + nt).
__device__ __forceinline__ bool level_work(int pairs, int rank, int round, int& pair, int& t0,
                                           int& nt) {
  if (pairs >= 4) {
    pair = rank + 4 * round;
    t0 = 0;
    nt = 4;
    return pair < pairs;
  }
  if (round > 0) return false;
  const int per = 4 / pairs;  // CTAs per combine
  pair = rank / per;
  nt = 4 / per;
  t0 = (rank % per) * nt;
  return true;
}

// Copy column tile `tile` (0, 1: M columns; 2, 3: D columns) of a package: src_m / src_d are
// the source's M and D pieces (both null: the identity package (I, 0)), dst the destination
// package ([M | D] contiguous).
__device__ void tile_copy(const float* src_m, const float* src_d, float* dst, int tile) {
  const bool mtile = tile < DK / NT;
  const int col0 = (mtile ? tile : tile - DK / NT) * NT;
  float* d = dst + (mtile ? 0 : DK * DK);
  const float* sp = mtile ? src_m : src_d;
  // 8 float4 per thread (256 threads): all loads before the first store
  float4 x[8];
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const int e = threadIdx.x + u * kThreads;
    const int r = e / (NT / 4), c4 = col0 + (e % (NT / 4)) * 4;
    if (sp) {
      x[u] = *reinterpret_cast<const float4*>(sp + r * DK + c4);
    } else {
      x[u] = make_float4(mtile && r == c4 ? 1.f : 0.f, mtile && r == c4 + 1 ? 1.f : 0.f,
                         mtile && r == c4 + 2 ? 1.f : 0.f, mtile && r == c4 + 3 ? 1.f : 0.f);
    }
  }
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const int e = threadIdx.x + u * kThreads;
    *reinterpret_cast<float4*>(d + (e / (NT / 4)) * DK + col0 + (e % (NT / 4)) * 4) = x[u];
  }
}
__device__ __forceinline__ void tile_move(const float* src, float* dst, int tile) {
  tile_copy(src, src + DK * DK, dst, tile);
}

__global__ void __cluster_dims__(4, 1, 1) __launch_bounds__(256, 1)
scan_tree_tc(Tree t, const int32_t* seq_off, const float* M, const float* D, const float* init,
             float* seg_init, float* final_state, uint32_t* status) {
  __shared__ uint64_t bar;
  __shared__ uint32_t tslot;
  const int tile = blockIdx.x, h = blockIdx.y, s = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5;
  if (warp == 0) {
    tmem_alloc(&tslot, NT);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  TileCtx cx{tslot, &bar, 0u, true};
  int first, cnt;
  if (!t.seq_range(seq_off, s, first, cnt) && tile == 0 && h == 0 && tid == 0 && status)
    atomicOr(status, KDA_STATUS_BAD_OFFSETS);
  const int64_t sd = (int64_t)DK * DK;
  // fill: packages of the sequence, then (I, 0)
  for (int i = 0; i < t.P2; ++i) {
    float* dst = t.node(s, i, h);
    if (i < cnt) {
      const float* m = M + ((int64_t)(first + i) * t.H + h) * sd;
      const float* d = D + ((int64_t)(first + i) * t.H + h) * sd;
      tile_copy(m, d, dst, tile);  // the caller's M and D arrays
    } else {
      tile_copy(nullptr, nullptr, dst, tile);
    }
  }
  cluster_sync_all();
  // up-sweep: a[i] = a[i] o a[i - d], written in place: every CTA working on a combine has its
  // A operand (a[i].M) in shared memory before any of them writes (the cluster barrier), and no
  // combine of the level reads another's a[i]
  const int rank = tile;
  for (int d = 1; d < t.P2; d <<= 1) {
    const int pairs = t.P2 / (2 * d);
    for (int round = 0; round * 4 < pairs || round == 0; ++round) {
      int pair, t0, nt;
      const bool mine = level_work(pairs, rank, round, pair, t0, nt);
      const int i = (2 * pair + 2) * d - 1;
      if (mine) load_a(t.node(s, i, h));
      __syncthreads();
      cluster_sync_all();
      if (mine) {
        float* A = t.node(s, i, h);
        const float* B = t.node(s, i - d, h);
        for (int tt = t0; tt < t0 + nt; ++tt)
          tile_product(cx, A + sd, B, B + sd, A, A + sd, tt, status);
      }
      cluster_sync_all();
    }
  }
  // root: the exit state (D tiles), then (I, 0)
  float* root = t.node(s, t.P2 - 1, h);
  if (final_state && tile >= DK / NT) {
    float* fo = final_state + ((int64_t)s * t.H + h) * sd;
    load_a(root);
    __syncthreads();
    tile_product(cx, root + sd, nullptr, init ? init + ((int64_t)s * t.H + h) * sd : nullptr,
                 nullptr, fo, tile, status);
  }
  cluster_sync_all();
  tile_copy(nullptr, nullptr, root, tile);
  cluster_sync_all();
  // down-sweep: (a[i - d], a[i]) <- (a[i], a[i - d] o a[i]); the combines go to tmp nodes,
  // then each CTA moves the tiles it computed
  for (int d = t.P2 / 2; d >= 1; d >>= 1) {
    const int pairs = t.P2 / (2 * d);
    for (int round = 0; round * 4 < pairs || round == 0; ++round) {
      int pair, t0, nt;
      if (level_work(pairs, rank, round, pair, t0, nt)) {
        const int i = (2 * pair + 2) * d - 1;
        const float* A = t.node(s, i - d, h);
        const float* B = t.node(s, i, h);
        float* o = t.tnode(s, pair, h);
        load_a(A);
        __syncthreads();
        for (int tt = t0; tt < t0 + nt; ++tt)
          tile_product(cx, A + sd, B, B + sd, o, o + sd, tt, status);
      }
    }
    cluster_sync_all();
    for (int round = 0; round * 4 < pairs || round == 0; ++round) {
      int pair, t0, nt;
      if (!level_work(pairs, rank, round, pair, t0, nt)) continue;
      const int i = (2 * pair + 2) * d - 1;
      for (int tt = t0; tt < t0 + nt; ++tt) {
        tile_move(t.node(s, i, h), t.node(s, i - d, h), tt);
        tile_move(t.tnode(s, pair, h), t.node(s, i, h), tt);
      }
    }
    cluster_sync_all();
  }
  // entry states: leaf j's prefix applied to the sequence's entry state, both D tiles of a
  // leaf by one CTA (its prefix's M loaded once)
  for (int j = rank; j < cnt; j += 4) {
    const float* pre = t.node(s, j, h);
    float* so = seg_init + ((int64_t)(first + j) * t.H + h) * sd;
    load_a(pre);
    __syncthreads();
    for (int dt = DK / NT; dt < 2 * (DK / NT); ++dt)
      tile_product(cx, pre + sd, nullptr, init ? init + ((int64_t)s * t.H + h) * sd : nullptr,
                   nullptr, so, dt, status);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tslot, NT);
}

}  // namespace tc

// ------------------------------------------------------------ sequential chain
// For the segment counts of real prompts (a 2048-token segment floor gives tens of segments per
// sequence) the plain left fold is the faster schedule: S_0 = S_init, seg_init[j] = S_j,
// S_{j+1} = M_j S_j + D_j, final = S_cnt, one dependent 128 x 128 x 128 product per segment
// (the tree has 2 log2 P dependent levels, each a heavier product spread over only 4 CTAs).
// The columns of the state are independent, so a CTA owns 64 of them and needs nothing from
// another CTA. Per step, on tcgen05 in 3xTF32 (A = M_j from TMEM, B = S_j from shared memory):
//   * warps 8..11 stream M_j in K-blocks of 32 columns into a ring of 3 TMEM slots (hi and lo
//     parts), each block as soon as the MMAs that read its slot's last occupant are done, so
//     the next step's operand is in place before its state is;
//   * warps 0..7 read the accumulator, add D_j, write S_{j+1} out (seg_init or the final state)
//     and store its hi / lo parts transposed as the next B operand; then one thread issues the
//     next step's 48 MMAs.
namespace seqtc {

using namespace ptx;

constexpr int DK = 128;
constexpr int NT = 64;                       // state columns per CTA
constexpr int kThreads = 384;                // 8 state warps + 4 M warps
constexpr uint32_t B_KB = NT * 128;          // B operand K-block: 64 rows x 128 B
constexpr uint32_t BH = 0, BL = 4 * B_KB;
// per-warp staging of a 32-row x 128-byte tile (12 warps x 4 KiB), 128-byte swizzle: global
// memory is read and written in whole 512-byte runs, each thread's row in shared memory
constexpr uint32_t STG = 8 * B_KB;
constexpr uint32_t SMEM = STG + 12 * 4096 + 1024;  // + alignment slack
constexpr int kSlots = 3;                    // TMEM ring of M K-blocks
constexpr uint32_t TM_ACC = 0, TM_SLOT = NT, kTmemCols = 256;
static_assert(TM_SLOT + kSlots * 64 <= kTmemCols, "TMEM overflow");

__device__ __forceinline__ float hi(float x) {
  return __uint_as_float(__float_as_uint(x) & 0xFFFFE000u);
}

// Tile of 32 rows x 32 floats (row stride `ld` floats) between global memory and a warp's
// staging buffer: lane l moves rows 4u + l / 8, 16-byte chunk l % 8 (coalesced); then each lane
// owns row l. The 128-byte swizzle keeps both access patterns free of bank conflicts.
__device__ __forceinline__ uint32_t stg_off(int row, int chunk) {
  return (uint32_t)row * 128u + ((uint32_t)(chunk ^ (row & 7)) << 4);
}
__device__ __forceinline__ void tile_ld(const float* src, int64_t ld, int lane, float4* g) {
#pragma unroll
  for (int u = 0; u < 8; ++u)
    g[u] = *reinterpret_cast<const float4*>(src + (int64_t)(4 * u + (lane >> 3)) * ld +
                                            (lane & 7) * 4);
}
__device__ __forceinline__ void stage_in(uint8_t* stg, const float4* g, int lane) {
#pragma unroll
  for (int u = 0; u < 8; ++u)
    *reinterpret_cast<float4*>(stg + stg_off(4 * u + (lane >> 3), lane & 7)) = g[u];
}
__device__ __forceinline__ void row_out(const uint8_t* stg, int lane, float* v) {
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const float4 x = *reinterpret_cast<const float4*>(stg + stg_off(lane, u));
    v[4 * u] = x.x; v[4 * u + 1] = x.y; v[4 * u + 2] = x.z; v[4 * u + 3] = x.w;
  }
}
__device__ __forceinline__ void row_in(uint8_t* stg, int lane, const float* v) {
#pragma unroll
  for (int u = 0; u < 8; ++u)
    *reinterpret_cast<float4*>(stg + stg_off(lane, u)) =
        make_float4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
}
__device__ __forceinline__ void tile_st(float* dst, int64_t ld, int lane, const uint8_t* stg) {
#pragma unroll
  for (int u = 0; u < 8; ++u)
    *reinterpret_cast<float4*>(dst + (int64_t)(4 * u + (lane >> 3)) * ld + (lane & 7) * 4) =
        *reinterpret_cast<const float4*>(stg + stg_off(4 * u + (lane >> 3), lane & 7));
}

// Named barrier 1 over the 256 state threads; returns whether any of them passed true.
__device__ __forceinline__ bool state_bar_or(bool x) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "bar.red.or.pred p, 1, 256, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)x)
      : "memory");
  return r != 0;
}

__global__ void __launch_bounds__(kThreads, 1)
scan_seq_tc(const int32_t* seq_off, int n_segs, int max_segs, int H, const float* M,
            const float* D, const float* init, float* seg_init, float* final_state,
            uint32_t* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  __shared__ uint64_t full[kSlots], empty[kSlots], acc_bar, drain;
  __shared__ uint32_t tslot;
  __shared__ int abort_flag;
  const int tile = blockIdx.x, h = blockIdx.y, s = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int q = warp & 3;
  const int r = q * 32 + lane;  // row of the state (and of M) this thread's TMEM lane holds
  const uint32_t lane_base = (uint32_t)(q * 32) << 16;
  if (warp == 0) {
    tmem_alloc(&tslot, kTmemCols);
    tmem_relinquish();
  }
  if (tid == 0) {
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(&full[i], 4);
      mbar_init(&empty[i], 1);
    }
    mbar_init(&acc_bar, 1);
    mbar_init(&drain, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tslot;
  const uint32_t sbase = smem_u32(sm);
  uint8_t* stg = sm + STG + warp * 4096;

  int first = seq_off[s], cnt = seq_off[s + 1] - first;
  if (first < 0 || cnt < 0 || cnt > max_segs || first + cnt > n_segs) {
    if (tile == 0 && h == 0 && tid == 0 && status) atomicOr(status, KDA_STATUS_BAD_OFFSETS);
    first = 0;
    cnt = 0;
  }
  const int64_t sd = (int64_t)DK * DK;
  auto fail = [&]() {
    abort_flag = 1;
    if (status) atomicOr(status, KDA_STATUS_TIMEOUT);
  };

  if (warp < 8) {
    // ------------------------------------------------ state warps: row r, 32 columns
    const int cb = (warp >> 2) * 32;
    const int col = tile * NT + cb;  // first global state column of this thread
    auto ld8 = [&](const float* src, float* v) {
      const float4* p = reinterpret_cast<const float4*>(src);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const float4 x = p[u];
        v[4 * u] = x.x; v[4 * u + 1] = x.y; v[4 * u + 2] = x.z; v[4 * u + 3] = x.w;
      }
    };
    // a state (or D) tile of this warp: rows 32 q .., columns col .. col + 31
    const int64_t toff = (int64_t)(q * 32) * DK + col;
    auto put = [&](float* base, const float* v) {  // v = this lane's row -> global, coalesced
      __syncwarp();
      row_in(stg, lane, v);
      __syncwarp();
      tile_st(base + toff, DK, lane, stg);
    };
    auto get_d = [&](int seg, float* d) {  // D_seg's tile -> this lane's row
      float4 g[8];
      tile_ld(D + ((int64_t)seg * H + h) * sd + toff, DK, lane, g);
      __syncwarp();
      stage_in(stg, g, lane);
      __syncwarp();
      row_out(stg, lane, d);
    };
    // B = S (row n = state column, K = state row r), split hi / lo, transposed
    auto store_b = [&](const float* v) {
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const uint32_t off = sw128_off32((uint32_t)(cb + j), (uint32_t)r, B_KB);
        const float hh = hi(v[j]);
        *reinterpret_cast<float*>(sm + BH + off) = hh;
        *reinterpret_cast<float*>(sm + BL + off) = v[j] - hh;
      }
    };
    auto issue = [&](int j) {  // one thread: S_{j+1} = M_j S_j in the accumulator
      const uint32_t idesc = idesc_make(kFmtTF32, 128, NT, false, false);
      const uint64_t dbh = sdesc_sw128(sbase + BH, 16, 1024);
      const uint64_t dbl = sdesc_sw128(sbase + BL, 16, 1024);
#pragma unroll
      for (int kb = 0; kb < 4; ++kb) {
        const int b = 4 * j + kb, slot = b % kSlots, use = b / kSlots;
        if (!mbar_wait_relaxed_or(&full[slot], (uint32_t)use & 1u, &abort_flag)) {
          fail();
          return;
        }
        tc_fence_after();
        const uint32_t a = tbase + TM_SLOT + (uint32_t)slot * 64u;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          const uint64_t bh = desc_add(dbh, kb * B_KB + ks * 32);
          const uint64_t bl = desc_add(dbl, kb * B_KB + ks * 32);
          mma_tf32_ts(tbase + TM_ACC, a + ks * 8, bh, idesc, (kb | ks) != 0 ? 1u : 0u);
          mma_tf32_ts(tbase + TM_ACC, a + ks * 8, bl, idesc, 1u);
          mma_tf32_ts(tbase + TM_ACC, a + 32 + ks * 8, bh, idesc, 1u);
        }
        mma_commit(&empty[slot]);
      }
      mma_commit(&acc_bar);
    };
    float v[32], d[32];
    if (init) {
      ld8(init + ((int64_t)s * H + h) * sd + (int64_t)r * DK + col, v);
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = 0.0f;
    }
    if (cnt == 0) {
      if (final_state) put(final_state + ((int64_t)s * H + h) * sd, v);
    } else {
      put(seg_init + ((int64_t)first * H + h) * sd, v);
      store_b(v);
      fence_proxy_async_smem();
      tc_fence_before();
      state_bar_or(false);
      tc_fence_after();
      if (tid == 0) issue(0);
      get_d(first, d);
      for (int j = 0; j < cnt; ++j) {
        __syncwarp();
        bool ok = mbar_wait_relaxed_or(&acc_bar, (uint32_t)j & 1u, &abort_flag);
        ok = __all_sync(0xFFFFFFFFu, ok);
        tc_fence_after();
        const bool last = j + 1 == cnt;
        if (ok) {
          tmem_ld32(tbase + lane_base + TM_ACC + cb, v);
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] += d[e];
          if (!last) {
            store_b(v);
            fence_proxy_async_smem();
          }
        } else if (lane == 0) {
          fail();
        }
        tc_fence_before();
        const bool stop = state_bar_or(!ok);
        tc_fence_after();
        if (stop) break;
        if (!last && tid == 0) issue(j + 1);
        float* out = last ? (final_state ? final_state + ((int64_t)s * H + h) * sd : nullptr)
                          : seg_init + ((int64_t)(first + j + 1) * H + h) * sd;
        if (out) put(out, v);
        if (!last) get_d(first + j + 1, d);
      }
    }
  } else if (cnt > 0) {
    // ------------------------------------------------ M warps: row r, K-blocks of 32 columns
    const int nb = 4 * cnt;
    auto ldm = [&](int b, float4* x) {  // block b of this warp's 32 rows, coalesced
      tile_ld(M + ((int64_t)(first + b / 4) * H + h) * sd + (int64_t)(q * 32) * DK + (b & 3) * 32,
              DK, lane, x);
    };
    // three register buffers in fixed roles (the loop is unrolled by three so that no buffer
    // is copied: a copy would wait for its loads), each block's loads two blocks ahead
    float4 buf[3][8];
    ldm(0, buf[0]);
    if (nb > 1) ldm(1, buf[1]);
    bool stop = false;
    for (int b0 = 0; b0 < nb && !stop; b0 += kSlots) {
#pragma unroll
      for (int k = 0; k < kSlots; ++k) {
        const int b = b0 + k;  // block b goes to slot k (kSlots = 3 divides b0)
        if (b >= nb || stop) break;
        if (b + 2 < nb) ldm(b + 2, buf[(k + 2) % kSlots]);
        const int use = b / kSlots;
        if (use > 0 && !mbar_wait_relaxed_or(&empty[k], (uint32_t)(use - 1) & 1u, &abort_flag)) {
          if (lane == 0) fail();
          stop = true;
          break;
        }
        tc_fence_after();
        float xh[32], xl[32];
        __syncwarp();
        stage_in(stg, buf[k], lane);
        __syncwarp();
        row_out(stg, lane, xl);  // row r of the block
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          xh[c] = hi(xl[c]);
          xl[c] -= xh[c];
        }
        const uint32_t a = tbase + lane_base + TM_SLOT + (uint32_t)k * 64u;
        tmem_st32_nowait(a, xh);
        tmem_st32_nowait(a + 32, xl);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_relaxed(&full[k]);
      }
    }
  }
  // every MMA this CTA issued has completed before TMEM is freed
  if (tid == 0) {
    mma_commit(&drain);
    if (!mbar_wait(&drain, 0) && status) atomicOr(status, KDA_STATUS_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tbase, kTmemCols);
}

}  // namespace seqtc

// Sequences of at most this many segments take the sequential chain (one product per segment);
// longer ones the tree.
constexpr int kSeqScanMaxSegs = 256;
constexpr int DK_TILES_SEQ = 128 / seqtc::NT;

int next_pow2(int x) {
  int p = 1;
  while (p < x) p <<= 1;
  return p;
}

// dk = dv = 128 on tensor cores. Same tree and same kernels for fill / reset / copies.
kda_status run_tc(int n_seqs, int n_segs, const int32_t* seq_off, int max_segs, int H,
                  const float* M, const float* D, const float* init, float* seg_init,
                  float* final_state, void* ws, uint32_t* status, cudaStream_t s) {
  constexpr int DK = 128, DV = 128;
  Tree t;
  t.P2 = next_pow2(max_segs);
  t.H = H;
  t.dk = DK;
  t.dv = DV;
  t.n_segs = n_segs;
  t.max_segs = max_segs;
  t.base = (float*)ws;
  t.tmp = t.base + (int64_t)n_seqs * t.P2 * H * pkg_floats(DK, DV);
  const int smem = (int)tc::SMEM;
  cudaFuncSetAttribute(tc::scan_tree_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  tc::scan_tree_tc<<<dim3(4, H, n_seqs), 256, smem, s>>>(t, seq_off, M, D, init, seg_init,
                                                          final_state, status);
  count_launches(1);
  return check_launch("kda_package_scan (tensor cores)");
}

template <int DK, int DV>
kda_status run(int n_seqs, int n_segs, const int32_t* seq_off, int max_segs, int H,
               const float* M,
               const float* D, const float* init, float* seg_init, float* final_state,
               void* ws, uint32_t* status, cudaStream_t s) {
  Tree t;
  t.P2 = next_pow2(max_segs);
  t.H = H;
  t.dk = DK;
  t.dv = DV;
  t.n_segs = n_segs;
  t.max_segs = max_segs;
  t.base = (float*)ws;
  t.tmp = t.base + (int64_t)n_seqs * t.P2 * H * pkg_floats(DK, DV);
  const int rb = DK / kRows;
  scan_fill<<<dim3(t.P2, H, n_seqs), kThreads, 0, s>>>(t, M, D, seq_off, status);
  for (int d = 1; d < t.P2; d <<= 1)
    scan_up<DK, DV><<<dim3(t.P2 / (2 * d), H * rb, n_seqs), kThreads, 0, s>>>(t, d);
  scan_root<DK, DV><<<dim3(1, H * rb, n_seqs), kThreads, 0, s>>>(t, init, final_state);
  for (int d = t.P2 / 2; d >= 1; d >>= 1) {
    scan_down_combine<DK, DV><<<dim3(t.P2 / (2 * d), H * rb, n_seqs), kThreads, 0, s>>>(t, d);
    scan_down_move<<<dim3(t.P2 / (2 * d), H, n_seqs), kThreads, 0, s>>>(t, d);
  }
  scan_apply<DK, DV><<<dim3(t.P2, H * rb, n_seqs), kThreads, 0, s>>>(t, seq_off, init,
                                                                      seg_init);
  int levels = 0;
  for (int d = 1; d < t.P2; d <<= 1) ++levels;
  count_launches(3 + 3 * levels);
  return check_launch("kda_package_scan");
}

}  // namespace

size_t scan_workspace_bytes(int n_seqs, int max_segs, int H, int dk, int dv) {
  const int64_t P2 = next_pow2(max_segs < 1 ? 1 : max_segs);
  const int64_t nodes = (int64_t)n_seqs * (P2 + P2 / 2) * H;
  return (size_t)(nodes * pkg_floats(dk, dv) * sizeof(float)) + 256;
}

kda_status launch_scan(int n_seqs, int n_segs, const int32_t* seq_seg_offsets, int max_segs,
                       int H, int dk, int dv, const float* M, const float* D,
                       const float* init_state, float* seg_init, float* final_state,
                       void* ws, size_t ws_bytes, uint32_t* status, cudaStream_t s) {
  (void)ws_bytes;
  if (n_seqs == 0) return KDA_OK;
  if (dk == 128 && dv == 128 && max_segs <= kSeqScanMaxSegs && n_seqs <= 65535 &&
      H <= 65535) {
    const int smem = (int)seqtc::SMEM;
    cudaFuncSetAttribute(seqtc::scan_seq_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    seqtc::scan_seq_tc<<<dim3(DK_TILES_SEQ, H, n_seqs), seqtc::kThreads, smem, s>>>(
        seq_seg_offsets, n_segs, max_segs, H, M, D, init_state, seg_init, final_state, status);
    count_launches(1);
    return check_launch("kda_package_scan (sequential, tensor cores)");
  }
  if (dk == 128 && dv == 128 && (int64_t)n_seqs * H <= 65535)
    return run_tc(n_seqs, n_segs, seq_seg_offsets, max_segs, H, M, D, init_state, seg_init,
                  final_state, ws, status, s);
  if (dk == 128 && dv == 128)
    return run<128, 128>(n_seqs, n_segs, seq_seg_offsets, max_segs, H, M, D, init_state, seg_init,
                         final_state, ws, status, s);
  if (dk == 64 && dv == 64)
    return run<64, 64>(n_seqs, n_segs, seq_seg_offsets, max_segs, H, M, D, init_state, seg_init,
                       final_state, ws, status, s);
  return set_error(KDA_ERR_UNSUPPORTED, "kda_package_scan: dk = dv must be 64 or 128");
}

}  // namespace kda
