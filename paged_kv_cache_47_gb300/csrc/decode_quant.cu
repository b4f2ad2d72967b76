// Split-K decode kernel variants for 8-bit caches (int8 / E4M3 codes with
// per-row scales; see decode_kernel.cuh). head_dim 128, tensor-core math.
#include "decode_kernel.cuh"

namespace pkv {

const DecodeVariant *find_variant_quant(int code_dtype, int act_dtype, int D, int gmax) {
    if (D != 128) return nullptr;
    if (act_dtype == PKV_F16) {
        using T = __half;
        if (code_dtype == PKV_INT8)
            return gmax == 8 ? SplitVariant<T, 128, 8, true, kQuantInt8>::get()
                             : SplitVariant<T, 128, 16, true, kQuantInt8>::get();
        return gmax == 8 ? SplitVariant<T, 128, 8, true, kQuantE4m3>::get()
                         : SplitVariant<T, 128, 16, true, kQuantE4m3>::get();
    }
    using T = __nv_bfloat16;
    if (code_dtype == PKV_INT8)
        return gmax == 8 ? SplitVariant<T, 128, 8, true, kQuantInt8>::get()
                         : SplitVariant<T, 128, 16, true, kQuantInt8>::get();
    return gmax == 8 ? SplitVariant<T, 128, 8, true, kQuantE4m3>::get()
                     : SplitVariant<T, 128, 16, true, kQuantE4m3>::get();
}

}  // namespace pkv
