// fp32 instantiations of the paged decode kernel (CUDA-core path): G = 1, 2 and
// the run-time-group kernel for the other group sizes.
#include "pa_decode.cuh"

namespace pa {

template <int D, int BS>
static void pick(int group, DecodeVariant* out) {
    switch (group) {
        case 1: *out = VariantOf<float, D, BS, false, 1>::get(); break;
        case 2: *out = VariantOf<float, D, BS, false, 2>::get(); break;
        default: *out = VariantOf<float, D, BS, false, 0>::get(); break;
    }
}

bool decode_variant_f32(int head_dim, int block_size, int group, DecodeVariant* out) {
    if (group == 4 || group == 8) return decode_variant_f32_pow2(head_dim, block_size, group, out);
    if (head_dim == 128 && block_size == 16) return pick<128, 16>(group, out), true;
    if (head_dim == 128 && block_size == 32) return pick<128, 32>(group, out), true;
    if (head_dim == 64 && block_size == 16) return pick<64, 16>(group, out), true;
    if (head_dim == 64 && block_size == 32) return pick<64, 32>(group, out), true;
    return false;
}

}  // namespace pa
