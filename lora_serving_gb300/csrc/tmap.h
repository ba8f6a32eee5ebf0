// tmap.h -- host-side encoding of TMA tensor maps (2-D, bf16, row-major).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace lora {

// A 2-D bf16 tensor of `rows` rows x `cols` columns with a row stride of
// `ld` elements (ld >= cols, ld * 2 a multiple of 16 bytes, base 16-byte
// aligned), read in boxes of box_rows x box_cols.  128-byte swizzle needs
// box_cols == 64.  Out-of-range box elements read as zero.  Returns false
// if the driver rejects the description.
bool encode_tmap_bf16(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint64_t ld,
                      uint32_t box_rows, uint32_t box_cols, bool swizzle128);

// A 3-D bf16 tensor [n2][n1][n0] (n0 innermost, strides ld1 and ld2
// elements for dimensions 1 and 2) read in 128-byte-swizzled boxes of
// box0 (= 64) x 1 x box2.  Elements past n0 read as zero, which pads a
// short innermost extent inside a longer stored row.
bool encode_tmap_bf16_3d(CUtensorMap* map, const void* base, uint64_t n0, uint64_t n1, uint64_t n2, uint64_t ld1,
                         uint64_t ld2, uint32_t box0, uint32_t box2);

}  // namespace lora
