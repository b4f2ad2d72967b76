// Split-K decode kernel variants for 8-bit caches (int8 / E4M3 codes with
// per-row scales; see decode_kernel.cuh). head_dim 128, tensor-core math:
// mma.sync for int8 and for E4M3 units of more than 8 heads, tcgen05 for
// E4M3 units of up to 4 or 8 heads.
#include "decode_kernel.cuh"

namespace pkv {

// gmax: 4 (E4M3 only), 8 or 16 heads per unit
template <typename T>
static const DecodeVariant *quant_variant(int code_dtype, int gmax) {
    if (code_dtype == PKV_INT8)
        return gmax <= 8 ? SplitVariant<T, 128, 8, true, kQuantInt8>::get()
                         : SplitVariant<T, 128, 16, true, kQuantInt8>::get();
    return gmax == 4   ? SplitVariant<T, 128, 4, true, kQuantE4m3>::get()
           : gmax == 8 ? SplitVariant<T, 128, 8, true, kQuantE4m3>::get()
                       : SplitVariant<T, 128, 16, true, kQuantE4m3>::get();
}

const DecodeVariant *find_variant_quant(int code_dtype, int act_dtype, int D, int gmax) {
    if (D != 128) return nullptr;
    return act_dtype == PKV_F16 ? quant_variant<__half>(code_dtype, gmax)
                                : quant_variant<__nv_bfloat16>(code_dtype, gmax);
}

}  // namespace pkv
