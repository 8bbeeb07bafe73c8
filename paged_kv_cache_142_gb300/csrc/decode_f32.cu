// fp32 instantiations of the paged decode kernel.
#include "decode_kernel.cuh"

namespace pa {

bool decode_info_f32(int head_dim, int group, DecodeKernelInfo* info) {
  using T = float;
#define PA_CASE(D, G)                 \
  if (head_dim == D && group == G) {  \
    fill_info<T, D, G>(info);         \
    return true;                      \
  }
  PA_CASE(64, 1) PA_CASE(64, 2) PA_CASE(64, 4) PA_CASE(64, 8)
  PA_CASE(128, 1) PA_CASE(128, 2) PA_CASE(128, 4) PA_CASE(128, 8)
#undef PA_CASE
  return false;
}

}  // namespace pa
