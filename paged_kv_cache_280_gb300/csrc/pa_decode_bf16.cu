// bf16 instantiations of the paged decode kernel on the tensor-core path (G >= 4).
#include "pa_decode.cuh"

namespace pa {

bool decode_variant_bf16_mma(int head_dim, int block_size, DecodeVariant* out) {
    using T = __nv_bfloat16;
#define PA_CASE(D_, BS_)                                       \
    if (head_dim == D_ && block_size == BS_) {                 \
        *out = VariantOf<T, D_, BS_, true, 0>::get();          \
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
