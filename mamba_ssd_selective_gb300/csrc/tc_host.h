// Host-side helpers shared by the tensor-core translation units: cached TMA
// tensor maps of token-major bf16 and float32 tensors and the device's compute capability.
// Not part of the public ABI.
#pragma once
#include <cuda.h>
#include <stdint.h>

namespace ssd {

// (inner, rows, batch) view of a [B, L, inner] bf16 tensor, box (box_cols, box_rows, 1):
// 64 columns with the 128-byte swizzle or 32 columns with the 64-byte swizzle;
// encoded once per (pointer, shape, box) and cached.
bool tma_map_tokens(CUtensorMap *out, const void *base, int64_t inner, int64_t L, int64_t B, int box_rows,
                    int box_cols = 64);

// (inner, rows, batch) view of a [B, L, inner] float32 tensor, box (box_cols, box_rows, 1):
// 32 columns with the 128-byte swizzle or 16 with the 64-byte swizzle (for TMA
// stores of float32 results).
bool tma_map_tokens_f32(CUtensorMap *out, const void *base, int64_t inner, int64_t L, int64_t B, int box_rows,
                        int box_cols = 32);

// Major compute capability of the current device (cached per device), -1 if unknown.
int device_cc_major_cached();

}  // namespace ssd
