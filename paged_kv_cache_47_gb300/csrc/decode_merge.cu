// Log-sum-exp merge launcher (kernel in decode_kernel.cuh).
#include "decode_kernel.cuh"

namespace pkv {

cudaError_t launch_merge(const DecodeParams &p, int D, cudaStream_t st) {
    if (p.C <= 1) return cudaSuccess;  // a single CTA finishes every unit itself
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(p.C - 1));
    cfg.blockDim = dim3(kMergeThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (D == 64) return cudaLaunchKernelEx(&cfg, decode_merge_kernel<64>, p);
    return cudaLaunchKernelEx(&cfg, decode_merge_kernel<128>, p);
}

}  // namespace pkv
