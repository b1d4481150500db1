#include "common.cuh"
#include "head_tc.h"

namespace df2 {

bool head_tc_supported(int64_t, int64_t, int64_t, int) { return false; }
size_t head_tc_workspace(int64_t, int64_t, int64_t, int, int) { return 0; }
int head_tc_launch(const uint16_t*, int64_t, int64_t, const uint16_t*, int64_t, int, const uint16_t*,
                   int, float*, int32_t*, float*, void*, int32_t*, int, cudaStream_t) {
    return DF2_ERR_UNSUPPORTED;
}

}  // namespace df2
