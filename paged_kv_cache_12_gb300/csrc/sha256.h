// SHA-256 of a byte string (FIPS 180-4), used for the chained block hashes.
#pragma once
#include <cstddef>
#include <cstdint>

namespace pa {
void sha256(const uint8_t *data, size_t n, uint8_t out[32]);
}
