// Instantiations of the tensor-core paged decode kernel (bf16, head_dim 128),
// one kv head per item; decode_umma_kh2.cu holds the two-kv-head items.
#include "decode_umma.cuh"

namespace pa {

const void* decode_umma_kh2_fn(int group);

const void* decode_umma_fn(int group, int kv_per_item) {
  if (kv_per_item == 2) return decode_umma_kh2_fn(group);
  if (kv_per_item != 1) return nullptr;
  switch (group) {
    case 1: return reinterpret_cast<const void*>(&paged_decode_umma_kernel<1, 1>);
    case 2: return reinterpret_cast<const void*>(&paged_decode_umma_kernel<2, 1>);
    case 4: return reinterpret_cast<const void*>(&paged_decode_umma_kernel<4, 1>);
    case 8: return reinterpret_cast<const void*>(&paged_decode_umma_kernel<8, 1>);
    case 16: return reinterpret_cast<const void*>(&paged_decode_umma_kernel<16, 1>);
    default: return nullptr;
  }
}

}  // namespace pa
