// Tensor-core (tcgen05 + TMEM + TMA) chunkwise KDA prefill for bf16 inputs.
#pragma once

#include <string>

#include "../../include/kda.h"
#include "kda_chunk_simt.cuh"

namespace kda {

inline bool tc_supports(int C) { return false; }

inline kda_status_t launch_chunk_tc(const SeqParams&, int, int, cudaStream_t, std::string& err) {
  err = "tensor-core path not built";
  return KDA_ERR_UNSUPPORTED;
}

}  // namespace kda
