// fp32 instantiations of the paged decode kernel (CUDA-core path): G = 4 and 8.
#include "pa_decode.cuh"

namespace pa {

template <int D, int BS>
static void pick(int group, DecodeVariant* out) {
    if (group == 4)
        *out = VariantOf<float, D, BS, false, 4>::get();
    else
        *out = VariantOf<float, D, BS, false, 8>::get();
}

bool decode_variant_f32_pow2(int head_dim, int block_size, int group, DecodeVariant* out) {
    if (group != 4 && group != 8) return false;
    if (head_dim == 128 && block_size == 16) return pick<128, 16>(group, out), true;
    if (head_dim == 128 && block_size == 32) return pick<128, 32>(group, out), true;
    if (head_dim == 64 && block_size == 16) return pick<64, 16>(group, out), true;
    if (head_dim == 64 && block_size == 32) return pick<64, 32>(group, out), true;
    return false;
}

}  // namespace pa
