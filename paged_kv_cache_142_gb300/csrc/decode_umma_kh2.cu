// Instantiations of the tensor-core paged decode kernel with two kv heads per
// work item (bf16, head_dim 128, GQA group 1, 2 or 4, blocks of 8..64 tokens).
#include "decode_umma.cuh"

namespace pa {

const void* decode_umma_kh2_fn(int group) {
  switch (group) {
    case 1: return reinterpret_cast<const void*>(&paged_decode_umma_kernel<1, 2>);
    case 2: return reinterpret_cast<const void*>(&paged_decode_umma_kernel<2, 2>);
    case 4: return reinterpret_cast<const void*>(&paged_decode_umma_kernel<4, 2>);
    default: return nullptr;
  }
}

}  // namespace pa
