#include "internal.h"
#include "ptx.cuh"
namespace stt {
size_t attn_bwd_workspace(int B, int H, int Q_LEN) { return ((size_t)B * H * Q_LEN * 4 + 15) / 16 * 16; }
cudaError_t attn_bwd_launch(const AttnArgs&, const AttnBwdArgs&, cudaStream_t) { return cudaErrorNotSupported; }
STT_DEFINE_ERROR_ACCESSOR(attn_bwd_error_word)
}
