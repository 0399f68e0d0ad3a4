// Tensor-core chunk kernel (tcgen05 + TMEM + TMA) for bf16 inputs.
#include "kda_internal.cuh"

namespace kda {

bool chunk_tc_supported(const ChunkParams& p, kda_dtype dt) {
  (void)p;
  (void)dt;
  return false;
}

kda_status launch_chunk_tc(const ChunkParams& p, kda_dtype dt, cudaStream_t s) {
  (void)p;
  (void)dt;
  (void)s;
  return set_error(KDA_ERR_UNSUPPORTED, "tensor-core chunk kernel: not available");
}

}  // namespace kda
