// SHA-256 (FIPS 180-4) for prefix-cache block keys.
#pragma once

#include <cstddef>
#include <cstdint>

#include "pa.h"

namespace pa {

class Sha256 {
 public:
  Sha256();
  void update(const void* data, size_t n);
  void finish(uint8_t out[32]);  // once; the object is spent afterwards

 private:
  uint32_t h_[8];
  uint8_t buf_[64];
  size_t fill_ = 0;
  uint64_t bytes_ = 0;
};

}  // namespace pa
