// CUDA-core window attention, fp32 instantiations.
#include "attn_simt.cuh"

namespace wedlm {

cudaError_t AttnVariants<float>::launch(int dpt, dim3 g, int th, size_t sm,
                                        cudaStream_t st, const AttnArgs& A) {
  switch (dpt) {
    case 4: attn_simt_kernel<float, 4><<<g, th, sm, st>>>(A); break;
    case 8: attn_simt_kernel<float, 8><<<g, th, sm, st>>>(A); break;
    case 16: attn_simt_kernel<float, 16><<<g, th, sm, st>>>(A); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

template cudaError_t launch_attention<float>(const AttnArgs&, cudaStream_t);
template cudaError_t launch_attention_merge<float>(const AttnArgs&, cudaStream_t);

}  // namespace wedlm
