// Split-KV merge for bf16 contexts (their attention runs on the tensor
// cores, k_attn_tc.cu; the merge is shared with the CUDA-core path).
#include "attn_simt.cuh"

namespace wedlm {

template cudaError_t launch_attention_merge<bf16>(const AttnArgs&, cudaStream_t);

}  // namespace wedlm
