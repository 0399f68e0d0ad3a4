// kda_package_scan_noalloc: the package scan with its scratch in a fixed device array that
// ships with the library, for callers that cannot allocate device memory.
//
// Who needs this: hosts that drive the library from a code path where allocating is not an
// option, e.g. a serving loop that has reserved all of HBM up front for its state pools (a
// cudaMalloc there fails, or must first evict something) or a custom-op interface that hands
// the op its inputs and outputs but no allocator. kda_package_scan needs a workspace of
// kda_package_scan_workspace(...) bytes from its caller; this variant uses the array below
// instead and allocates nothing: no cudaMalloc, no cudaFree, no allocating library routine.
//
// The array: kNoAllocScratchBytes (64 MiB) of device memory, 256-byte aligned, reserved on
// every GPU that loads this library's device code and held until the process exits. Calls
// whose scan needs more than that are rejected with KDA_ERR_WORKSPACE. All calls share the
// one array, and it keeps the last call's contents; the scan writes every byte it reads
// before reading it, so nothing needs clearing between calls. Calls whose work overlaps on
// the GPU (different streams, or different host threads without ordering) race on it.
//
// The device address of the array is looked up once per device, on the first call made with
// that device current (host code cannot pass the array's name to a kernel: in host code the
// name is a stand-in, not a device address). Make that first call before any stream capture.
// The cached address belongs to the device's current context: after cudaDeviceReset the
// array lives at a new address and this entry point must not be called again in that process.
#include <mutex>
#include <string>

#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_scan_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_scan_scratch on the current device (looked up once per device).
kda_status scratch_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess)
    return set_error(KDA_ERR_CUDA, std::string("kda_package_scan_noalloc: cudaGetDevice: ") +
                                       cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices)
    return set_error(KDA_ERR_UNSUPPORTED, "kda_package_scan_noalloc: device index >= 64");
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_scan_scratch);
    if (e != cudaSuccess || !p)
      return set_error(KDA_ERR_CUDA,
                       std::string("kda_package_scan_noalloc: cudaGetSymbolAddress: ") +
                           cudaGetErrorString(e));
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return KDA_OK;
}

}  // namespace
}  // namespace kda

using namespace kda;

extern "C" KDA_API kda_status kda_package_scan_noalloc(
    int n_seqs, int n_segs, const int32_t* seq_seg_offsets, int max_segs_per_seq, int H,
    int dk, int dv, const float* M, const float* D, const float* init_state, float* seg_init,
    float* final_state, uint32_t* status, kda_stream_t stream) {
  const char* fn = "kda_package_scan_noalloc";
  if (H <= 0) return set_error(KDA_ERR_INVALID_ARG, std::string(fn) + ": H must be > 0");
  if (!((dk == 64 && dv == 64) || (dk == 128 && dv == 128)))
    return set_error(KDA_ERR_UNSUPPORTED, std::string(fn) + ": dk = dv must be 64 or 128");
  if (n_seqs < 0 || n_segs < 0)
    return set_error(KDA_ERR_INVALID_ARG, std::string(fn) + ": n_seqs and n_segs must be >= 0");
  if (n_seqs == 0) return KDA_OK;
  if (max_segs_per_seq < 1 || max_segs_per_seq > 65536)
    return set_error(KDA_ERR_INVALID_ARG,
                     std::string(fn) + ": max_segs_per_seq must be in [1, 65536]");
  const size_t need = scan_workspace_bytes(n_seqs, max_segs_per_seq, H, dk, dv);
  if (need > kNoAllocScratchBytes)
    return set_error(KDA_ERR_WORKSPACE,
                     std::string(fn) + ": this scan needs " + std::to_string(need) +
                         " bytes of scratch; the built-in array holds " +
                         std::to_string(kNoAllocScratchBytes) +
                         " (use kda_package_scan with a caller workspace)");
  void* ws = nullptr;
  kda_status st = scratch_address(&ws);
  if (st != KDA_OK) return st;
  st = kda_package_scan(n_seqs, n_segs, seq_seg_offsets, max_segs_per_seq, H, dk, dv, M, D,
                        init_state, seg_init, final_state, ws, kNoAllocScratchBytes, status,
                        stream);
  if (st != KDA_OK) {  // report the failure under this entry point's name
    std::string m = kda_last_error();
    const std::string inner = "kda_package_scan";
    if (m.rfind(inner, 0) == 0) m = std::string(fn) + m.substr(inner.size());
    return set_error(st, m);
  }
  return st;
}
