// Split-K decode kernel variants for the prefix-aware decode (see
// decode_kernel.cuh, PFX = true): fp16 / bf16 paged caches, tensor-core math.
#include "decode_kernel.cuh"

namespace pkv {

template <typename T>
const DecodeVariant *prefix_variant(int D, int gmax) {
    if (D == 64) return gmax == 8 ? SplitVariant<T, 64, 8, true, 0, false, false, true>::get()
                                  : SplitVariant<T, 64, 16, true, 0, false, false, true>::get();
    if (D == 128) return gmax == 8 ? SplitVariant<T, 128, 8, true, 0, false, false, true>::get()
                                   : SplitVariant<T, 128, 16, true, 0, false, false, true>::get();
    return nullptr;
}

const DecodeVariant *find_variant_prefix(int dtype, int D, int gmax) {
    if (gmax != 8 && gmax != 16) return nullptr;
    if (dtype == PKV_F16) return prefix_variant<__half>(D, gmax);
    if (dtype == PKV_BF16) return prefix_variant<__nv_bfloat16>(D, gmax);
    return nullptr;
}

}  // namespace pkv
