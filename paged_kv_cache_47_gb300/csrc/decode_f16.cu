// Split-K decode kernel variants for f16 K/V (see decode_kernel.cuh).
#include "decode_kernel.cuh"

namespace pkv {

const DecodeVariant *find_variant_f16(int D, int gmax, bool mma) {
    using T = __half;
    if (mma) {
        if (D == 64 && gmax == 8) return SplitVariant<T, 64, 8, true>::get();
        if (D == 64 && gmax == 16) return SplitVariant<T, 64, 16, true>::get();
        if (D == 128 && gmax == 8) return SplitVariant<T, 128, 8, true>::get();
        if (D == 128 && gmax == 16) return SplitVariant<T, 128, 16, true>::get();
        return nullptr;
    }
    if (D == 64 && gmax == 1) return SplitVariant<T, 64, 1, false>::get();
    if (D == 64 && gmax == 2) return SplitVariant<T, 64, 2, false>::get();
    if (D == 64 && gmax == 4) return SplitVariant<T, 64, 4, false>::get();
    if (D == 64 && gmax == 8) return SplitVariant<T, 64, 8, false>::get();
    if (D == 64 && gmax == 16) return SplitVariant<T, 64, 16, false>::get();
    if (D == 128 && gmax == 1) return SplitVariant<T, 128, 1, false>::get();
    if (D == 128 && gmax == 2) return SplitVariant<T, 128, 2, false>::get();
    if (D == 128 && gmax == 4) return SplitVariant<T, 128, 4, false>::get();
    if (D == 128 && gmax == 8) return SplitVariant<T, 128, 8, false>::get();
    if (D == 128 && gmax == 16) return SplitVariant<T, 128, 16, false>::get();
    return nullptr;
}

}  // namespace pkv
