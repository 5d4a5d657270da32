// Decode over FP8 (E4M3) pools with bf16 queries and outputs, on the tensor
// cores for every group size: the K and V codes are widened to f16 in
// registers and the MMAs run in f16 (a group of fewer than 8 query heads pads
// the MMA's N).  head_dim 128: one pool row is one 128-byte swizzle panel.
#include "pa_decode.cuh"

namespace pa {

template <int BS>
static bool pick(DecodeVariant* out) {
    *out = VariantOf<__nv_bfloat16, 128, BS, true, 0, __nv_fp8_e4m3>::get();
    return true;
}

bool decode_variant_fp8(int head_dim, int block_size, int group, DecodeVariant* out) {
    if (head_dim != 128) return false;
    if (block_size == 16) return pick<16>(out);
    if (block_size == 32) return pick<32>(out);
    return false;
}

}  // namespace pa
