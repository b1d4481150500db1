// Tensor-core (tcgen05/TMEM, TMA-fed) unary logits + top-K + hidden projection.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "kernels.h"

namespace df2 {

bool head_tc_supported(int64_t P, int64_t D, int64_t V, int K);
size_t head_tc_workspace(int64_t P, int64_t D, int64_t V, int K, int num_sms);
// stall_stage >= 0 (self-test only): that pipeline stage's copies are never
// issued, so the kernel's bounded waits time out and report it in dev_status.
// parts_out != null: the per-CTA lists are left in the workspace for the caller
// to fold (ids/vals are not written).  zero_words[0 .. n_zero): set to zero by the
// kernel, for counters the next kernel in the stream expects at zero.
int head_tc_launch(const uint16_t* h, int64_t P, int64_t D, const uint16_t* W, int64_t V, int K,
                   const uint16_t* W_H, int r, float* G, int32_t* ids, float* vals, void* ws,
                   int32_t* dev_status, int num_sms, cudaStream_t stream, int stall_stage = -1,
                   TopkParts* parts_out = nullptr, unsigned* zero_words = nullptr, int n_zero = 0);

}  // namespace df2
