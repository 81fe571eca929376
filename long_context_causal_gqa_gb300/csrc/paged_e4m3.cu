// paged_e4m3.cu -- placeholder launcher; the kernel is added separately.
#include "internal.h"

namespace gqa {

size_t paged_e4m3_workspace_bytes(int R, int ctx_len, int num_sms) {
    (void)R;
    (void)ctx_len;
    (void)num_sms;
    return kWorkspaceCounterBytes;
}

int paged_e4m3_launch(const void*, const uint8_t*, const uint8_t*, const float*, const float*,
                      const int32_t*, int, int, int, float, void*, cudaStream_t) {
    return GQA_ERR_UNSUPPORTED;
}

int sparse_launch(const void*, const void*, const void*, const int32_t*, const int32_t*,
                  const int32_t*, int, int, int, int, float, void*, cudaStream_t) {
    return GQA_ERR_UNSUPPORTED;
}

}  // namespace gqa
