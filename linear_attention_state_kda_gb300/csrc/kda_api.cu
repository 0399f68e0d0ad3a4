// C-ABI entry points of libkda.so: host-side argument checks, then one launch sequence on
// the caller's stream. See include/kda.h for the contract of each call.
#include <atomic>
#include <cstdio>
#include <string>

#include "kda_internal.cuh"

namespace kda {

static thread_local std::string g_last_error;
static std::atomic<uint64_t> g_launches{0};

void count_launches(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

kda_status set_error(kda_status st, const std::string& msg) {
  g_last_error = msg;
  return st;
}

kda_status check_launch(const char* what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess)
    return set_error(KDA_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
  return KDA_OK;
}

namespace {

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

kda_status check_shape(const char* fn, kda_dtype dt, int H, int dk, int dv, int chunk) {
  if (dt != KDA_F32 && dt != KDA_BF16)
    return set_error(KDA_ERR_UNSUPPORTED, std::string(fn) + ": dtype must be KDA_F32 or KDA_BF16");
  if (H <= 0) return set_error(KDA_ERR_INVALID_ARG, std::string(fn) + ": H must be > 0");
  if (!((dk == 64 && dv == 64) || (dk == 128 && dv == 128)))
    return set_error(KDA_ERR_UNSUPPORTED, std::string(fn) + ": dk = dv must be 64 or 128");
  if (chunk != kChunk)
    return set_error(KDA_ERR_UNSUPPORTED, std::string(fn) + ": chunk must be 64");
  return KDA_OK;
}

#define KDA_REQUIRE(cond, st, msg)           \
  do {                                       \
    if (!(cond)) return set_error(st, msg);  \
  } while (0)

size_t chunk_workspace(kda_dtype dt, int n_ranges, int total_tokens, int H, int dk, int dv) {
  if (n_ranges <= 0 || total_tokens <= 0 || H <= 0) return 0;
  if (!chunk_tc_shape_ok(dt, n_ranges, total_tokens, H, dk, dv)) return 0;
  return chunk_tc_workspace_bytes(n_ranges, total_tokens, H);
}

// A shape with a positive workspace query runs on the tensor-core kernels and nowhere else:
// if they cannot run (the driver lacks the tensor-map encoder), the call fails.
kda_status chunked(const char* fn, const ChunkParams& p, kda_dtype dt, void* ws, size_t ws_bytes,
                   cudaStream_t s) {
  const size_t need = chunk_workspace(dt, p.n_ranges, p.total_tokens, p.H, p.dk, p.dv);
  if (need == 0) return launch_chunk_simt(p, dt, s);
  KDA_REQUIRE(ws && ws_bytes >= need && aligned(ws, 256), KDA_ERR_WORKSPACE,
              std::string(fn) + ": workspace missing, too small or not 256-byte aligned (need " +
                  std::to_string(need) + " bytes)");
  KDA_REQUIRE(chunk_tc_available(), KDA_ERR_UNSUPPORTED,
              std::string(fn) + ": the CUDA driver does not provide cuTensorMapEncodeTiled, "
                                "which the tensor-core path needs");
  return launch_chunk_tc(p, dt, ws, ws_bytes, s);
}

}  // namespace
}  // namespace kda

using namespace kda;

extern "C" {

const char* kda_last_error(void) { return g_last_error.c_str(); }

const char* kda_version(void) { return "kda-gb300 0.1 (sm_103a)"; }

uint64_t kda_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

size_t kda_chunk_workspace(kda_dtype dt, int n_ranges, int total_tokens, int H, int dk, int dv) {
  return chunk_workspace(dt, n_ranges, total_tokens, H, dk, dv);
}

kda_status kda_chunk_prefill(kda_dtype dt, int n_seqs, int total_tokens,
                             const int32_t* cu_seqlens, int H, int dk, int dv, int chunk,
                             float scale, const void* q, const void* k, const void* v,
                             const float* g, const float* beta, const float* init_state,
                             void* o, float* final_state, void* workspace, size_t ws_bytes,
                             uint32_t* status, kda_stream_t stream) {
  const char* fn = "kda_chunk_prefill";
  kda_status st = check_shape(fn, dt, H, dk, dv, chunk);
  if (st != KDA_OK) return st;
  KDA_REQUIRE(n_seqs >= 0 && total_tokens >= 0, KDA_ERR_INVALID_ARG,
              "kda_chunk_prefill: n_seqs and total_tokens must be >= 0");
  KDA_REQUIRE(cu_seqlens || n_seqs <= 1, KDA_ERR_INVALID_ARG,
              "kda_chunk_prefill: cu_seqlens is required when n_seqs > 1");
  if (n_seqs == 0) return KDA_OK;
  KDA_REQUIRE(total_tokens == 0 || (q && k && v && g && beta && o), KDA_ERR_INVALID_ARG,
              "kda_chunk_prefill: q, k, v, g, beta and o must be non-null");
  KDA_REQUIRE(aligned(q, 16) && aligned(k, 16) && aligned(v, 16) && aligned(o, 16) &&
                  aligned(g, 16) && aligned(beta, 16) && aligned(init_state, 16) &&
                  aligned(final_state, 16) && aligned(cu_seqlens, 4) && aligned(status, 4),
              KDA_ERR_INVALID_ARG,
              "kda_chunk_prefill: q, k, v, g, beta, o and the states must be 16-byte aligned");
  ChunkParams p{};
  p.q = q; p.k = k; p.v = v; p.g = g; p.beta = beta;
  p.offsets = cu_seqlens; p.n_ranges = n_seqs; p.total_tokens = total_tokens;
  p.H = H; p.dk = dk; p.dv = dv; p.scale = scale;
  p.init = init_state; p.o = o; p.final_state = final_state; p.status = status;
  p.package = 0;
  return chunked(fn, p, dt, workspace, ws_bytes, (cudaStream_t)stream);
}

kda_status kda_segment_package(kda_dtype dt, int n_segs, int total_tokens,
                               const int32_t* seg_offsets, int H, int dk, int dv, int chunk,
                               const void* k, const void* v, const float* g,
                               const float* beta, float* M, float* D, void* workspace,
                               size_t ws_bytes, uint32_t* status, kda_stream_t stream) {
  const char* fn = "kda_segment_package";
  kda_status st = check_shape(fn, dt, H, dk, dv, chunk);
  if (st != KDA_OK) return st;
  KDA_REQUIRE(n_segs >= 0 && total_tokens >= 0, KDA_ERR_INVALID_ARG,
              "kda_segment_package: n_segs and total_tokens must be >= 0");
  if (n_segs == 0) return KDA_OK;
  KDA_REQUIRE(seg_offsets && M && D, KDA_ERR_INVALID_ARG,
              "kda_segment_package: seg_offsets, M and D must be non-null");
  KDA_REQUIRE(total_tokens == 0 || (k && v && g && beta), KDA_ERR_INVALID_ARG,
              "kda_segment_package: k, v, g and beta must be non-null");
  KDA_REQUIRE(aligned(k, 16) && aligned(v, 16) && aligned(g, 16) && aligned(beta, 16) &&
                  aligned(M, 16) && aligned(D, 16) && aligned(seg_offsets, 4) &&
                  aligned(status, 4),
              KDA_ERR_INVALID_ARG,
              "kda_segment_package: k, v, g, beta, M and D must be 16-byte aligned");
  ChunkParams p{};
  p.k = k; p.v = v; p.g = g; p.beta = beta;
  p.offsets = seg_offsets; p.n_ranges = n_segs; p.total_tokens = total_tokens;
  p.H = H; p.dk = dk; p.dv = dv; p.scale = 1.0f;
  p.M = M; p.D = D; p.status = status; p.package = 1;
  return chunked(fn, p, dt, workspace, ws_bytes, (cudaStream_t)stream);
}

size_t kda_package_scan_workspace(int n_seqs, int max_segs_per_seq, int H, int dk, int dv) {
  if (n_seqs <= 0 || max_segs_per_seq <= 0 || H <= 0 || dk <= 0 || dv <= 0) return 0;
  return scan_workspace_bytes(n_seqs, max_segs_per_seq, H, dk, dv);
}

kda_status kda_package_scan(int n_seqs, int n_segs, const int32_t* seq_seg_offsets,
                            int max_segs_per_seq, int H, int dk, int dv, const float* M,
                            const float* D, const float* init_state, float* seg_init,
                            float* final_state, void* workspace, size_t ws_bytes,
                            uint32_t* status, kda_stream_t stream) {
  KDA_REQUIRE(H > 0, KDA_ERR_INVALID_ARG, "kda_package_scan: H must be > 0");
  KDA_REQUIRE((dk == 64 && dv == 64) || (dk == 128 && dv == 128), KDA_ERR_UNSUPPORTED,
              "kda_package_scan: dk = dv must be 64 or 128");
  KDA_REQUIRE(n_seqs >= 0 && n_segs >= 0, KDA_ERR_INVALID_ARG,
              "kda_package_scan: n_seqs and n_segs must be >= 0");
  if (n_seqs == 0) return KDA_OK;
  KDA_REQUIRE(max_segs_per_seq >= 1 && max_segs_per_seq <= 65536, KDA_ERR_INVALID_ARG,
              "kda_package_scan: max_segs_per_seq must be in [1, 65536]");
  KDA_REQUIRE(seq_seg_offsets && (n_segs == 0 || (M && D && seg_init)), KDA_ERR_INVALID_ARG,
              "kda_package_scan: seq_seg_offsets, M, D and seg_init must be non-null");
  KDA_REQUIRE(aligned(M, 16) && aligned(D, 16) && aligned(seg_init, 16) &&
                  aligned(init_state, 16) && aligned(final_state, 16) &&
                  aligned(seq_seg_offsets, 4) && aligned(status, 4),
              KDA_ERR_INVALID_ARG, "kda_package_scan: pointers must be 16-byte aligned");
  const size_t need = scan_workspace_bytes(n_seqs, max_segs_per_seq, H, dk, dv);
  KDA_REQUIRE(workspace && ws_bytes >= need && aligned(workspace, 256), KDA_ERR_WORKSPACE,
              "kda_package_scan: workspace missing, too small or not 256-byte aligned (need " +
                  std::to_string(need) + " bytes)");
  return launch_scan(n_seqs, n_segs, seq_seg_offsets, max_segs_per_seq, H, dk, dv, M, D,
                     init_state, seg_init, final_state, workspace, ws_bytes, status,
                     (cudaStream_t)stream);
}

kda_status kda_segment_replay(kda_dtype dt, int n_segs, int total_tokens,
                              const int32_t* seg_offsets, int H, int dk, int dv, int chunk,
                              float scale, const void* q, const void* k, const void* v,
                              const float* g, const float* beta, const float* seg_init,
                              void* o, float* seg_final, void* workspace, size_t ws_bytes,
                              uint32_t* status, kda_stream_t stream) {
  KDA_REQUIRE(n_segs == 0 || seg_offsets, KDA_ERR_INVALID_ARG,
              "kda_segment_replay: seg_offsets must be non-null");
  kda_status st = kda_chunk_prefill(dt, n_segs, total_tokens, seg_offsets, H, dk, dv, chunk,
                                    scale, q, k, v, g, beta, seg_init, o, seg_final, workspace,
                                    ws_bytes, status, stream);
  if (st != KDA_OK) {
    std::string m = g_last_error;
    if (m.rfind("kda_chunk_prefill", 0) == 0) m = "kda_segment_replay" + m.substr(17);
    return set_error(st, m);
  }
  return st;
}

kda_status kda_chunk_prepare(kda_dtype dt, int n_ranges, int total_tokens,
                             const int32_t* offsets, int H, int dk, int dv, int chunk,
                             float scale, const void* q, const void* k, const void* v,
                             const float* g, const float* beta, void* workspace,
                             size_t ws_bytes, uint32_t* status, kda_stream_t stream) {
  const char* fn = "kda_chunk_prepare";
  kda_status st = check_shape(fn, dt, H, dk, dv, chunk);
  if (st != KDA_OK) return st;
  KDA_REQUIRE(n_ranges >= 0 && total_tokens >= 0, KDA_ERR_INVALID_ARG,
              "kda_chunk_prepare: n_ranges and total_tokens must be >= 0");
  KDA_REQUIRE(offsets || n_ranges <= 1, KDA_ERR_INVALID_ARG,
              "kda_chunk_prepare: offsets are required when n_ranges > 1");
  if (n_ranges == 0 || total_tokens == 0) return KDA_OK;
  KDA_REQUIRE(chunk_workspace(dt, n_ranges, total_tokens, H, dk, dv) > 0, KDA_ERR_UNSUPPORTED,
              "kda_chunk_prepare: records exist for the tensor-core shapes only (bf16, "
              "dk = dv = 128, H a multiple of 4)");
  KDA_REQUIRE(k && v && g && beta, KDA_ERR_INVALID_ARG,
              "kda_chunk_prepare: k, v, g and beta must be non-null");
  KDA_REQUIRE(aligned(q, 16) && aligned(k, 16) && aligned(v, 16) && aligned(g, 16) &&
                  aligned(beta, 16) && aligned(offsets, 4) && aligned(status, 4),
              KDA_ERR_INVALID_ARG,
              "kda_chunk_prepare: q, k, v, g must be 16-byte aligned, beta too");
  ChunkParams p{};
  p.q = q; p.k = k; p.v = v; p.g = g; p.beta = beta;
  p.offsets = offsets; p.n_ranges = n_ranges; p.total_tokens = total_tokens;
  p.H = H; p.dk = dk; p.dv = dv; p.scale = scale; p.status = status;
  p.package = q ? 0 : 1;  // without q, only the factors a package walk reads
  const size_t need = chunk_workspace(dt, n_ranges, total_tokens, H, dk, dv);
  KDA_REQUIRE(workspace && ws_bytes >= need && aligned(workspace, 256), KDA_ERR_WORKSPACE,
              "kda_chunk_prepare: workspace missing, too small or not 256-byte aligned (need " +
                  std::to_string(need) + " bytes)");
  return launch_chunk_tc(p, dt, workspace, ws_bytes, (cudaStream_t)stream, kPhasePrep);
}

namespace {
kda_status check_prepared(const char* fn, kda_dtype dt, int n_segs, int total_tokens,
                          const int32_t* seg_offsets, int H, int dk, int dv, int chunk,
                          const void* workspace, size_t ws_bytes) {
  kda_status st = check_shape(fn, dt, H, dk, dv, chunk);
  if (st != KDA_OK) return st;
  KDA_REQUIRE(n_segs >= 0 && total_tokens >= 0, KDA_ERR_INVALID_ARG,
              std::string(fn) + ": n_segs and total_tokens must be >= 0");
  if (n_segs == 0 || total_tokens == 0) return KDA_OK;
  KDA_REQUIRE(seg_offsets, KDA_ERR_INVALID_ARG, std::string(fn) + ": seg_offsets must be non-null");
  const size_t need = chunk_workspace(dt, n_segs, total_tokens, H, dk, dv);
  KDA_REQUIRE(need > 0, KDA_ERR_UNSUPPORTED,
              std::string(fn) + ": prepared records exist for the tensor-core shapes only");
  KDA_REQUIRE(workspace && ws_bytes >= need && aligned(workspace, 256), KDA_ERR_WORKSPACE,
              std::string(fn) + ": workspace missing, too small or not 256-byte aligned");
  return KDA_OK;
}
}  // namespace

kda_status kda_segment_package_prepared(kda_dtype dt, int n_segs, int total_tokens,
                                        const int32_t* seg_offsets, int H, int dk, int dv,
                                        int chunk, float* M, float* D, const void* workspace,
                                        size_t ws_bytes, uint32_t* status, kda_stream_t stream) {
  const char* fn = "kda_segment_package_prepared";
  kda_status st = check_prepared(fn, dt, n_segs, total_tokens, seg_offsets, H, dk, dv, chunk,
                                 workspace, ws_bytes);
  if (st != KDA_OK || n_segs == 0) return st;
  KDA_REQUIRE(M && D && aligned(M, 16) && aligned(D, 16) && aligned(status, 4),
              KDA_ERR_INVALID_ARG, "kda_segment_package_prepared: M and D must be non-null and "
                                   "16-byte aligned");
  if (total_tokens == 0) return KDA_OK;
  ChunkParams p{};
  p.offsets = seg_offsets; p.n_ranges = n_segs; p.total_tokens = total_tokens;
  p.H = H; p.dk = dk; p.dv = dv; p.scale = 1.0f;
  p.M = M; p.D = D; p.status = status; p.package = 1;
  return launch_chunk_tc(p, dt, const_cast<void*>(workspace), ws_bytes, (cudaStream_t)stream,
                         kPhaseState);
}

kda_status kda_segment_replay_prepared(kda_dtype dt, int n_segs, int total_tokens,
                                       const int32_t* seg_offsets, int H, int dk, int dv,
                                       int chunk, const float* seg_init, void* o,
                                       float* seg_final, const void* workspace, size_t ws_bytes,
                                       uint32_t* status, kda_stream_t stream) {
  const char* fn = "kda_segment_replay_prepared";
  kda_status st = check_prepared(fn, dt, n_segs, total_tokens, seg_offsets, H, dk, dv, chunk,
                                 workspace, ws_bytes);
  if (st != KDA_OK || n_segs == 0 || total_tokens == 0) return st;
  KDA_REQUIRE(o && aligned(o, 16) && aligned(seg_init, 16) && aligned(seg_final, 16) &&
                  aligned(status, 4),
              KDA_ERR_INVALID_ARG, "kda_segment_replay_prepared: o must be non-null, pointers "
                                   "16-byte aligned");
  ChunkParams p{};
  p.offsets = seg_offsets; p.n_ranges = n_segs; p.total_tokens = total_tokens;
  p.H = H; p.dk = dk; p.dv = dv; p.scale = 1.0f;
  p.init = seg_init; p.o = o; p.final_state = seg_final; p.status = status; p.package = 0;
  return launch_chunk_tc(p, dt, const_cast<void*>(workspace), ws_bytes, (cudaStream_t)stream,
                         kPhaseState);
}

kda_status kda_debug_flag_wait(kda_dtype dt, int n_segs, int total_tokens,
                               const int32_t* seg_offsets, int H, int dk, int dv, int chunk,
                               const float* seg_init, void* o, float* seg_final,
                               const void* workspace, size_t ws_bytes, uint64_t limit_ns,
                               uint32_t* status, kda_stream_t stream) {
  const char* fn = "kda_debug_flag_wait";
  kda_status st = check_prepared(fn, dt, n_segs, total_tokens, seg_offsets, H, dk, dv, chunk,
                                 workspace, ws_bytes);
  if (st != KDA_OK || n_segs == 0 || total_tokens == 0) return st;
  KDA_REQUIRE(limit_ns >= 1000000ull && limit_ns <= 4000000000ull, KDA_ERR_INVALID_ARG,
              "kda_debug_flag_wait: limit_ns must be in [1e6, 4e9]");
  KDA_REQUIRE(o && aligned(o, 16) && aligned(seg_init, 16) && aligned(seg_final, 16) &&
                  aligned(status, 4),
              KDA_ERR_INVALID_ARG, "kda_debug_flag_wait: o must be non-null, pointers "
                                   "16-byte aligned");
  ChunkParams p{};
  p.offsets = seg_offsets; p.n_ranges = n_segs; p.total_tokens = total_tokens;
  p.H = H; p.dk = dk; p.dv = dv; p.scale = 1.0f;
  p.init = seg_init; p.o = o; p.final_state = seg_final; p.status = status; p.package = 0;
  p.flag_wait_ns = limit_ns;
  return launch_chunk_tc(p, dt, const_cast<void*>(workspace), ws_bytes, (cudaStream_t)stream,
                         kPhaseState | kPhaseFlags);
}

kda_status kda_decode_step(kda_dtype dt, int batch, int H, int dk, int dv, float scale,
                           const void* q, const void* k, const void* v, const float* g,
                           const float* beta, const int32_t* slot_ids, float* state_pool,
                           int64_t n_slots, void* o, uint32_t* status, kda_stream_t stream) {
  const char* fn = "kda_decode_step";
  kda_status st = check_shape(fn, dt, H, dk, dv, kChunk);
  if (st != KDA_OK) return st;
  KDA_REQUIRE(batch >= 0, KDA_ERR_INVALID_ARG, "kda_decode_step: batch must be >= 0");
  KDA_REQUIRE(n_slots > 0, KDA_ERR_INVALID_ARG, "kda_decode_step: n_slots must be > 0");
  if (batch == 0) return KDA_OK;
  KDA_REQUIRE(q && k && v && g && beta && slot_ids && state_pool && o, KDA_ERR_INVALID_ARG,
              "kda_decode_step: pointers must be non-null");
  KDA_REQUIRE((int64_t)batch * H <= (1LL << 30), KDA_ERR_INVALID_ARG,
              "kda_decode_step: batch * H must not exceed 2^30");
  KDA_REQUIRE(aligned(state_pool, 16) && aligned(q, 4) && aligned(k, 4) && aligned(v, 4) &&
                  aligned(o, 4) && aligned(g, 4) && aligned(beta, 4) && aligned(slot_ids, 4) &&
                  aligned(status, 4),
              KDA_ERR_INVALID_ARG, "kda_decode_step: misaligned pointer");
  return launch_decode(dt, batch, H, dk, dv, scale, q, k, v, g, beta, slot_ids, state_pool,
                       n_slots, o, status, (cudaStream_t)stream);
}

kda_status kda_decode_window(kda_dtype dt, int batch, int window, int H, int dk, int dv,
                             float scale, const void* q, const void* k, const void* v,
                             const float* g, const float* beta, unsigned flags,
                             const int32_t* read_slots, const int32_t* write_slots,
                             float* state_pool, int64_t n_slots, void* o, uint32_t* status,
                             kda_stream_t stream) {
  const char* fn = "kda_decode_window";
  kda_status st = check_shape(fn, dt, H, dk, dv, kChunk);
  if (st != KDA_OK) return st;
  KDA_REQUIRE(batch >= 0, KDA_ERR_INVALID_ARG, "kda_decode_window: batch must be >= 0");
  KDA_REQUIRE(window >= 0 && window <= kMaxWindow, KDA_ERR_UNSUPPORTED,
              "kda_decode_window: window must be in 0 .. 16");
  KDA_REQUIRE(n_slots > 0, KDA_ERR_INVALID_ARG, "kda_decode_window: n_slots must be > 0");
  KDA_REQUIRE((flags & ~KDA_DECODE_BETA_LOGIT) == 0, KDA_ERR_INVALID_ARG,
              "kda_decode_window: unknown flag bits");
  if (batch == 0 || window == 0) return KDA_OK;
  KDA_REQUIRE(q && k && v && g && beta && read_slots && write_slots && state_pool && o,
              KDA_ERR_INVALID_ARG, "kda_decode_window: pointers must be non-null");
  KDA_REQUIRE((int64_t)batch * window * H <= (1LL << 30), KDA_ERR_INVALID_ARG,
              "kda_decode_window: batch * window * H must not exceed 2^30");
  KDA_REQUIRE(aligned(state_pool, 16) && aligned(q, 4) && aligned(k, 4) && aligned(v, 4) &&
                  aligned(o, 4) && aligned(g, 4) && aligned(beta, 4) && aligned(read_slots, 4) &&
                  aligned(write_slots, 4) && aligned(status, 4),
              KDA_ERR_INVALID_ARG, "kda_decode_window: misaligned pointer");
  return launch_decode_window(dt, batch, window, H, dk, dv, scale, q, k, v, g, beta, flags,
                              read_slots, write_slots, state_pool, n_slots, o, status,
                              (cudaStream_t)stream);
}

kda_status kda_slot_zero(int n, const int32_t* slot_ids, float* state_pool, int64_t n_slots,
                         int64_t slot_elems, uint32_t* status, kda_stream_t stream) {
  KDA_REQUIRE(n >= 0 && n_slots > 0 && slot_elems >= 0, KDA_ERR_INVALID_ARG,
              "kda_slot_zero: n >= 0, n_slots > 0 and slot_elems >= 0 required");
  KDA_REQUIRE(slot_elems % 4 == 0, KDA_ERR_INVALID_ARG,
              "kda_slot_zero: slot_elems must be a multiple of 4");
  if (n == 0 || slot_elems == 0) return KDA_OK;
  KDA_REQUIRE(state_pool && aligned(state_pool, 16) && aligned(slot_ids, 4) &&
                  aligned(status, 4),
              KDA_ERR_INVALID_ARG, "kda_slot_zero: pool must be non-null and 16-byte aligned");
  KDA_REQUIRE(slot_ids || n <= n_slots, KDA_ERR_INVALID_ARG,
              "kda_slot_zero: without slot ids, n must not exceed n_slots");
  return launch_slots(true, n, nullptr, nullptr, 0, state_pool, slot_ids, n_slots, slot_elems,
                      status, (cudaStream_t)stream);
}

kda_status kda_slot_copy(int n, const float* src, const int32_t* src_ids, int64_t n_src,
                         float* dst, const int32_t* dst_ids, int64_t n_dst, int64_t slot_elems,
                         uint32_t* status, kda_stream_t stream) {
  KDA_REQUIRE(n >= 0 && n_src > 0 && n_dst > 0 && slot_elems >= 0, KDA_ERR_INVALID_ARG,
              "kda_slot_copy: n >= 0, n_src > 0, n_dst > 0 and slot_elems >= 0 required");
  KDA_REQUIRE(slot_elems % 4 == 0, KDA_ERR_INVALID_ARG,
              "kda_slot_copy: slot_elems must be a multiple of 4");
  if (n == 0 || slot_elems == 0) return KDA_OK;
  KDA_REQUIRE(src && dst && aligned(src, 16) && aligned(dst, 16) && aligned(src_ids, 4) &&
                  aligned(dst_ids, 4) && aligned(status, 4),
              KDA_ERR_INVALID_ARG, "kda_slot_copy: pools must be non-null and 16-byte aligned");
  KDA_REQUIRE((src_ids || n <= n_src) && (dst_ids || n <= n_dst), KDA_ERR_INVALID_ARG,
              "kda_slot_copy: without ids, n must not exceed that pool's slot count");
  return launch_slots(false, n, src, src_ids, n_src, dst, dst_ids, n_dst, slot_elems, status,
                      (cudaStream_t)stream);
}

kda_status kda_short_conv(kda_dtype dt, int n_seqs, int total_tokens, const int32_t* cu_seqlens,
                          int channels, int width, const void* x, const float* weight,
                          unsigned flags, const int32_t* read_slots, const int32_t* write_slots,
                          void* conv_state, int64_t n_slots, void* out, uint32_t* status,
                          kda_stream_t stream) {
  KDA_REQUIRE(dt == KDA_F32 || dt == KDA_BF16, KDA_ERR_UNSUPPORTED,
              "kda_short_conv: dtype must be KDA_F32 or KDA_BF16");
  KDA_REQUIRE(width >= 1 && width <= 4, KDA_ERR_UNSUPPORTED,
              "kda_short_conv: width must be in 1 .. 4");
  KDA_REQUIRE(channels > 0 && channels % 8 == 0, KDA_ERR_INVALID_ARG,
              "kda_short_conv: channels must be a positive multiple of 8");
  KDA_REQUIRE(n_seqs >= 0 && total_tokens >= 0, KDA_ERR_INVALID_ARG,
              "kda_short_conv: n_seqs and total_tokens must be >= 0");
  KDA_REQUIRE(cu_seqlens || n_seqs <= 1, KDA_ERR_INVALID_ARG,
              "kda_short_conv: cu_seqlens is required for more than one sequence");
  KDA_REQUIRE((flags & ~KDA_CONV_SILU) == 0, KDA_ERR_INVALID_ARG,
              "kda_short_conv: unknown flag bits");
  if (n_seqs == 0) return KDA_OK;
  const bool slots = (read_slots || write_slots) && width > 1;
  KDA_REQUIRE(!slots || (conv_state && n_slots > 0), KDA_ERR_INVALID_ARG,
              "kda_short_conv: slot tables need conv_state and n_slots > 0");
  KDA_REQUIRE(total_tokens == 0 || (x && weight && out), KDA_ERR_INVALID_ARG,
              "kda_short_conv: x, weight and out must be non-null");
  KDA_REQUIRE(((int64_t)total_tokens / 16 + n_seqs) * ((channels + 511) / 512) <= 0x7fffffffLL,
              KDA_ERR_INVALID_ARG, "kda_short_conv: too many tokens x channels for one launch");
  KDA_REQUIRE(aligned(x, 16) && aligned(out, 16) && aligned(conv_state, 16) &&
                  aligned(weight, 4) && aligned(cu_seqlens, 4) && aligned(read_slots, 4) &&
                  aligned(write_slots, 4) && aligned(status, 4),
              KDA_ERR_INVALID_ARG, "kda_short_conv: misaligned pointer");
  KDA_REQUIRE(!(x && x == out), KDA_ERR_INVALID_ARG, "kda_short_conv: out must not alias x");
  return launch_short_conv(dt, n_seqs, total_tokens, cu_seqlens, channels, width, x, weight,
                           flags, slots ? read_slots : nullptr, slots ? write_slots : nullptr,
                           conv_state, slots ? n_slots : 0, out, status, (cudaStream_t)stream);
}

}  // extern "C"
