// fp32 instantiations of the paged decode kernel (CUDA-core path).
#include "pa_decode.cuh"

namespace pa {

bool decode_variant_f32(int head_dim, int block_size, DecodeVariant* out) {
#define PA_CASE(D_, BS_)                                       \
    if (head_dim == D_ && block_size == BS_) {                 \
        *out = VariantOf<float, D_, BS_, false>::get();        \
        return true;                                           \
    }
    PA_CASE(128, 16)
    PA_CASE(128, 32)
    PA_CASE(64, 16)
    PA_CASE(64, 32)
#undef PA_CASE
    return false;
}

}  // namespace pa
