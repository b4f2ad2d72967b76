// Split-K decode kernel variants over flat per-sequence spans (see
// decode_kernel.cuh, FLAT = true): fp16 / bf16, tensor-core math.
#include "decode_kernel.cuh"

namespace pkv {

template <typename T>
const DecodeVariant *flat_variant(int D, int gmax) {
    if (D == 64) return gmax == 8 ? SplitVariant<T, 64, 8, true, 0, true>::get()
                                  : SplitVariant<T, 64, 16, true, 0, true>::get();
    if (D == 128) return gmax == 8 ? SplitVariant<T, 128, 8, true, 0, true>::get()
                                   : SplitVariant<T, 128, 16, true, 0, true>::get();
    return nullptr;
}

const DecodeVariant *find_variant_flat(int dtype, int D, int gmax) {
    if (dtype == PKV_F16) return flat_variant<__half>(D, gmax);
    if (dtype == PKV_BF16) return flat_variant<__nv_bfloat16>(D, gmax);
    return nullptr;
}

}  // namespace pkv
