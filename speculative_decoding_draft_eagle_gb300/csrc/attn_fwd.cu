#include "internal.h"
#include "ptx.cuh"
namespace stt {
cudaError_t attn_fwd_launch(const AttnArgs&, void*, float*, cudaStream_t) { return cudaErrorNotSupported; }
STT_DEFINE_ERROR_ACCESSOR(attn_fwd_error_word)
}
