// Split-K decode kernel variants with the append fused in (see
// decode_kernel.cuh, FUSED = true): fp16 / bf16 paged caches, tensor-core math.
#include "decode_kernel.cuh"

namespace pkv {

template <typename T>
const DecodeVariant *fused_variant(int D, int gmax) {
    if (D == 64) return gmax == 8 ? SplitVariant<T, 64, 8, true, 0, false, true>::get()
                                  : SplitVariant<T, 64, 16, true, 0, false, true>::get();
    if (D == 128) return gmax == 8 ? SplitVariant<T, 128, 8, true, 0, false, true>::get()
                                   : SplitVariant<T, 128, 16, true, 0, false, true>::get();
    return nullptr;
}

const DecodeVariant *find_variant_fused(int dtype, int D, int gmax) {
    if (gmax != 8 && gmax != 16) return nullptr;
    if (dtype == PKV_F16) return fused_variant<__half>(D, gmax);
    if (dtype == PKV_BF16) return fused_variant<__nv_bfloat16>(D, gmax);
    return nullptr;
}

}  // namespace pkv
