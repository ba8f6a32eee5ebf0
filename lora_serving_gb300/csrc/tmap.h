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

}  // namespace lora
