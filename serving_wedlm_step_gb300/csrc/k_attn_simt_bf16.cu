// CUDA-core window attention, bf16 instantiations (G*W rows up to 128 with 512 threads).
#include "attn_simt.cuh"

namespace wedlm {

cudaError_t AttnVariants<bf16>::launch(int dpt, dim3 g, int th, size_t sm,
                                        cudaStream_t st, const AttnArgs& A) {
  switch (dpt) {
    case 16: attn_simt_kernel<bf16, 16><<<g, th, sm, st>>>(A); break;
    case 32: attn_simt_kernel<bf16, 32><<<g, th, sm, st>>>(A); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

template cudaError_t launch_attention<bf16>(const AttnArgs&, cudaStream_t);
template cudaError_t launch_attention_merge<bf16>(const AttnArgs&, cudaStream_t);

}  // namespace wedlm
