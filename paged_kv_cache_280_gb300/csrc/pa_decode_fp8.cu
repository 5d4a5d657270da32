// Decode over FP8 (E4M3) pools with bf16 queries and outputs.  4 or more
// query heads per KV head take the tensor-core path (each stage's codes widened
// to f16 in shared memory, f16 mma.sync); 1-3 take the CUDA-core path (exact
// instantiations for 1 and 2, a run-time-group fallback for 3).  head_dim 128:
// one pool row is one 128-byte swizzle panel.
#include "pa_decode.cuh"

namespace pa {

template <int BS>
static bool pick(int group, DecodeVariant* out) {
    using T = __nv_bfloat16;
    using KV = __nv_fp8_e4m3;
    // 4+ query heads per KV head: the tensor-core path, each stage widened to f16 in shared memory
    if (group >= 4) {
        *out = VariantOf<T, 128, BS, true, 0, KV>::get();
        return true;
    }
    switch (group) {
        case 1: *out = VariantOf<T, 128, BS, false, 1, KV>::get(); return true;
        case 2: *out = VariantOf<T, 128, BS, false, 2, KV>::get(); return true;
        default: *out = VariantOf<T, 128, BS, false, 0, KV>::get(); return true;
    }
}

bool decode_variant_fp8(int head_dim, int block_size, int group, DecodeVariant* out) {
    if (head_dim != 128) return false;
    if (block_size == 16) return pick<16>(group, out);
    if (block_size == 32) return pick<32>(group, out);
    return false;
}

}  // namespace pa
