// Instantiations of the tensor-core paged decode kernel (bf16, head_dim 128).
#include "decode_umma.cuh"

namespace pa {

const void* decode_umma_fn(int group) {
  switch (group) {
    case 1: return reinterpret_cast<const void*>(&paged_decode_umma_kernel<1>);
    case 2: return reinterpret_cast<const void*>(&paged_decode_umma_kernel<2>);
    case 4: return reinterpret_cast<const void*>(&paged_decode_umma_kernel<4>);
    case 8: return reinterpret_cast<const void*>(&paged_decode_umma_kernel<8>);
    case 16: return reinterpret_cast<const void*>(&paged_decode_umma_kernel<16>);
    default: return nullptr;
  }
}

}  // namespace pa
