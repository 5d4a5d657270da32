// bf16 instantiations of the paged decode kernel on the CUDA-core path (G = 1, 2, 3).
#include "pa_decode.cuh"

namespace pa {

template <int D, int BS>
static bool pick(int group, DecodeVariant* out) {
    using T = __nv_bfloat16;
    switch (group) {
        case 1: *out = VariantOf<T, D, BS, false, 1>::get(); return true;
        case 2: *out = VariantOf<T, D, BS, false, 2>::get(); return true;
        case 3: *out = VariantOf<T, D, BS, false, 3>::get(); return true;
        default: return false;
    }
}

bool decode_variant_bf16_fma(int head_dim, int block_size, int group, DecodeVariant* out) {
    if (head_dim == 128 && block_size == 16) return pick<128, 16>(group, out);
    if (head_dim == 128 && block_size == 32) return pick<128, 32>(group, out);
    if (head_dim == 64 && block_size == 16) return pick<64, 16>(group, out);
    if (head_dim == 64 && block_size == 32) return pick<64, 32>(group, out);
    return false;
}

}  // namespace pa
