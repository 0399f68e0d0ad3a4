// Internal declarations shared by the translation units of libkda.so.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <string>

#include "../../include/kda.h"

namespace kda {

// Sets the thread-local message returned by kda_last_error() and passes the status through.
kda_status set_error(kda_status st, const std::string& msg);
kda_status check_launch(const char* what);
// Adds n to the process-wide launch counter returned by kda_launch_count().
void count_launches(int n);

// Per-token element access for the two input dtypes.
__device__ __forceinline__ float ld_elem(const float* p, int64_t i) { return p[i]; }
__device__ __forceinline__ float ld_elem(const __nv_bfloat16* p, int64_t i) {
  return __bfloat162float(p[i]);
}
__device__ __forceinline__ void st_elem(float* p, int64_t i, float x) { p[i] = x; }
__device__ __forceinline__ void st_elem(__nv_bfloat16* p, int64_t i, float x) {
  p[i] = __float2bfloat16_rn(x);
}

// One chunked pass over packed token ranges ("sequences": prefill sequences, replayed
// segments, or package segments). A CTA owns one (range, head, column tile).
//
// Column space: prefill/replay work on the dv value columns. Package mode works on the
// augmented state [M | D] (dk + dv columns): columns < dk start from the identity and see
// zero values, columns >= dk start from zero and see v.
struct ChunkParams {
  const void* q;          // [T, H, dk] (unused in package mode)
  const void* k;          // [T, H, dk]
  const void* v;          // [T, H, dv]
  const float* g;         // [T, H, dk]
  const float* beta;      // [T, H]
  const int32_t* offsets; // [n_ranges + 1] device, or nullptr: one range [0, total_tokens)
  int n_ranges, total_tokens, H, dk, dv;
  float scale;
  const float* init;      // [n_ranges, H, dk, dv] or nullptr (zeros)
  void* o;                // [T, H, dv] or nullptr
  float* final_state;     // [n_ranges, H, dk, dv] or nullptr
  float* M;               // package mode: [n_ranges, H, dk, dk]
  float* D;               // package mode: [n_ranges, H, dk, dv]
  uint32_t* status;       // optional device status word
  int package;            // 1 = package mode
  uint64_t flag_wait_ns;  // limit of a walk's wait for a record's ready flag (0: default)
  int discard;            // the walk drops each record's L2 lines once done (records private)
};

// Chunk size of every chunked kernel.
constexpr int kChunk = 64;
// Decay (nats over one chunk, per key channel) up to which the chunk kernels use the log-
// midpoint frame for that channel; a channel that decays more is computed frame-free.
constexpr float kMaxChunkDecay = 160.0f;

// FFMA (CUDA-core) chunk kernel: fp32 arithmetic throughout; any dtype.
kda_status launch_chunk_simt(const ChunkParams& p, kda_dtype dt, cudaStream_t s);

// Tensor-core (tcgen05/TMEM/TMA) chunk path for bf16 inputs with dk = dv = 128: a parallel
// per-(chunk, head) prep kernel writing workspace records, then the in-order state kernel.
// chunk_tc_shape_ok decides from shapes alone whether the path (and so the workspace)
// applies; chunk_tc_available tells whether the driver provides the tensor-map encoder the
// path needs.
bool chunk_tc_shape_ok(kda_dtype dt, int n_ranges, int total_tokens, int H, int dk, int dv);
size_t chunk_tc_workspace_bytes(int n_ranges, int total_tokens, int H);
bool chunk_tc_available();
// A row-major [rows][cols] array (bf16, or fp32 when f32) as a 2-D tensor map without swizzle,
// box [box_rows][box_cols]; false when the driver lacks the encoder or rejects the layout.
bool make_map_rows(CUtensorMap* m, const void* ptr, bool f32, uint64_t cols, uint64_t rows,
                   uint32_t box_cols, uint32_t box_rows);
// phases: kPhasePrep writes the records, kPhaseState walks them; both = one chunked call.
// kPhaseFlags (with kPhaseState alone) makes the walk wait for each record's ready flag in
// the workspace, as the fused launch's walk does (the flag-wait diagnostic).
constexpr int kPhasePrep = 1, kPhaseState = 2, kPhaseFlags = 4;
kda_status launch_chunk_tc(const ChunkParams& p, kda_dtype dt, void* workspace, size_t ws_bytes,
                           cudaStream_t s, int phases = kPhasePrep | kPhaseState);

// Decode step.
kda_status launch_decode(kda_dtype dt, int batch, int H, int dk, int dv, float scale,
                         const void* q, const void* k, const void* v, const float* g,
                         const float* beta, const int32_t* slot_ids, float* pool,
                         int64_t n_slots, void* o, uint32_t* status, cudaStream_t s);

// Verify window with a state fork (read slot, one write slot per window column).
constexpr int kMaxWindow = 16;
kda_status launch_decode_window(kda_dtype dt, int batch, int window, int H, int dk, int dv,
                                float scale, const void* q, const void* k, const void* v,
                                const float* g, const float* beta, unsigned flags,
                                const int32_t* read_slots, const int32_t* write_slots,
                                float* pool, int64_t n_slots, void* o, uint32_t* status,
                                cudaStream_t s);

// Whole-slot zero (zero = true; src unused) or copy src[src_ids[i]] -> dst[dst_ids[i]].
kda_status launch_slots(bool zero, int n, const float* src, const int32_t* src_ids, int64_t n_src,
                        float* dst, const int32_t* dst_ids, int64_t n_dst, int64_t slot_elems,
                        uint32_t* status, cudaStream_t s);

// Short causal depthwise convolution with per-sequence history windows (width 1..4).
kda_status launch_short_conv(kda_dtype dt, int n_seqs, int total, const int32_t* cu, int C,
                             int width, const void* x, const float* w, unsigned flags,
                             const int32_t* read_slots, const int32_t* write_slots, void* hist,
                             int64_t n_slots, void* out, uint32_t* status, cudaStream_t s);

// Package scan.
size_t scan_workspace_bytes(int n_seqs, int max_segs, int H, int dk, int dv);
kda_status launch_scan(int n_seqs, int n_segs, const int32_t* seq_seg_offsets, int max_segs,
                       int H, int dk, int dv, const float* M, const float* D,
                       const float* init_state, float* seg_init, float* final_state,
                       void* ws, size_t ws_bytes, uint32_t* status, cudaStream_t s);

}  // namespace kda
