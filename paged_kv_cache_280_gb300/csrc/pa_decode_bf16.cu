// bf16 instantiations of the paged decode kernel (tensor-core and CUDA-core paths).
#include "pa_decode.cuh"

namespace pa {

bool decode_variant_bf16(int head_dim, int block_size, bool mma, DecodeVariant* out) {
    using T = __nv_bfloat16;
#define PA_CASE(D_, BS_)                                                                         \
    if (head_dim == D_ && block_size == BS_) {                                                   \
        *out = mma ? VariantOf<T, D_, BS_, true>::get() : VariantOf<T, D_, BS_, false>::get(); \
        return true;                                                                             \
    }
    PA_CASE(128, 16)
    PA_CASE(128, 32)
    PA_CASE(64, 16)
    PA_CASE(64, 32)
#undef PA_CASE
    return false;
}

}  // namespace pa
