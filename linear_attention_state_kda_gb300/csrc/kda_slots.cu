// Whole-slot utilities over the fp32 state pool [n_slots, H, dk, dv]: zero a list of slots,
// and copy slots between two pools (or within one), which covers taking a checkpoint image
// of some slots into a compact buffer and restoring it.
//
// Sources: kern PR #44 ("Prefill-only pipeline parallelism, from kern cut to full Kimi-K3"),
// Runtime section (Runtime::zero_slot clears the state slot a new sequence is given); ATOM PR
// #2709 ("feat(kimi-k3): PP8 prefill for P/D serving - KDA state under PP"), sections on
// PAGE-backed KDA state checkpoints (a checkpoint image holds copies of a sequence's state,
// taken in stream order with the batch that produced it).
//
// Both are pure HBM streams (a 2 MiB slot at H = 32, d = 128). A CTA moves one contiguous
// 32 KiB span of one slot: each thread issues its 8 independent 16-byte loads before its
// stores, with streaming cache hints (the data is not reread). blockIdx.y walks the slot
// pairs, blockIdx.x the spans of a slot.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 8;
constexpr int kSpan = kThreads * kUnroll;  // float4 per CTA pass (32 KiB)

template <bool kZero>
__global__ void __launch_bounds__(kThreads)
slot_kernel(const float4* __restrict__ src, const int32_t* __restrict__ src_ids, int64_t n_src,
            float4* __restrict__ dst, const int32_t* __restrict__ dst_ids, int64_t n_dst, int n,
            int64_t slot_vec, uint32_t* status) {
  for (int pair = blockIdx.y; pair < n; pair += gridDim.y) {
    const int64_t di = dst_ids ? (int64_t)dst_ids[pair] : (int64_t)pair;
    const int64_t si = kZero ? 0 : (src_ids ? (int64_t)src_ids[pair] : (int64_t)pair);
    if (di >= n_dst || (!kZero && si >= n_src)) {
      if (blockIdx.x == 0 && threadIdx.x == 0 && status) atomicOr(status, KDA_STATUS_BAD_SLOT);
      continue;
    }
    if (di < 0 || si < 0) continue;
    float4* d = dst + di * slot_vec;
    const float4* s = kZero ? nullptr : src + si * slot_vec;
    for (int64_t base = (int64_t)blockIdx.x * kSpan; base < slot_vec;
         base += (int64_t)gridDim.x * kSpan) {
      float4 r[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int64_t i = base + u * kThreads + threadIdx.x;
        if constexpr (kZero) r[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        else if (i < slot_vec) r[u] = __ldcs(s + i);
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int64_t i = base + u * kThreads + threadIdx.x;
        if (i < slot_vec) __stcs(d + i, r[u]);
      }
    }
  }
}

}  // namespace

kda_status launch_slots(bool zero, int n, const float* src, const int32_t* src_ids, int64_t n_src,
                        float* dst, const int32_t* dst_ids, int64_t n_dst, int64_t slot_elems,
                        uint32_t* status, cudaStream_t s) {
  if (n == 0 || slot_elems == 0) return KDA_OK;
  const int64_t slot_vec = slot_elems / 4;
  const int64_t spans = (slot_vec + kSpan - 1) / kSpan;
  dim3 grid((unsigned)(spans < 65535 ? spans : 65535), (unsigned)(n < 65535 ? n : 65535));
  if (zero)
    slot_kernel<true><<<grid, kThreads, 0, s>>>(nullptr, nullptr, 0, (float4*)dst, dst_ids, n_dst,
                                                n, slot_vec, status);
  else
    slot_kernel<false><<<grid, kThreads, 0, s>>>((const float4*)src, src_ids, n_src, (float4*)dst,
                                                 dst_ids, n_dst, n, slot_vec, status);
  count_launches(1);
  return check_launch(zero ? "kda_slot_zero" : "kda_slot_copy");
}

}  // namespace kda
