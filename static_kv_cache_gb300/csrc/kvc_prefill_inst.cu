// kvc_prefill_inst.cu -- explicit chunked-prefill kernels for one 16-bit
// element type and head width, selected at compile time by KVC_INST_TYPE
// (0 bf16, 1 fp16) and KVC_INST_D (64 or 128).  The build compiles this file
// once per pair, in parallel.
#include "kvc_prefill.cuh"

#ifndef KVC_INST_TYPE
#error "KVC_INST_TYPE must be defined"
#endif
#ifndef KVC_INST_D
#error "KVC_INST_D must be defined"
#endif

#if KVC_INST_TYPE == 0
#define KVC_ELEM __nv_bfloat16
#define KVC_TAG bf16
#elif KVC_INST_TYPE == 1
#define KVC_ELEM __half
#define KVC_TAG f16
#else
#error "chunked prefill takes 16-bit caches"
#endif

#define KVC_PCAT2(a, b) prefill_kernel_##a##_##b
#define KVC_PCAT(a, b) KVC_PCAT2(a, b)
#define KVC_PTABLE_FN KVC_PCAT(KVC_TAG, KVC_INST_D)

namespace kvc {

const PrefillKernelInfo *KVC_PTABLE_FN(int G) {
    switch (G) {
        case 1: return prefill_info<KVC_ELEM, KVC_INST_D, 1>();
        case 2: return prefill_info<KVC_ELEM, KVC_INST_D, 2>();
        case 3: return prefill_info<KVC_ELEM, KVC_INST_D, 3>();
        case 4: return prefill_info<KVC_ELEM, KVC_INST_D, 4>();
        case 5: return prefill_info<KVC_ELEM, KVC_INST_D, 5>();
        case 6: return prefill_info<KVC_ELEM, KVC_INST_D, 6>();
        case 7: return prefill_info<KVC_ELEM, KVC_INST_D, 7>();
        case 8: return prefill_info<KVC_ELEM, KVC_INST_D, 8>();
        default: return nullptr;
    }
}

}  // namespace kvc
