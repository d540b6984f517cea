#pragma once
#include <cstddef>
#include <cstdint>

namespace cpr {
// FIPS 180-4 SHA-256 of `len` bytes.
void sha256(const void* data, size_t len, uint8_t out[32]);
}  // namespace cpr
