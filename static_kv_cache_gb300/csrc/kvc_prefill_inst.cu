// kvc_prefill_inst.cu -- explicit chunked-prefill kernels for one 16-bit
// element type and head width, selected at compile time by KVC_INST_TYPE
// (0 bf16, 1 fp16) and KVC_INST_D (64 or 128).  The build compiles this file
// once per pair, in parallel.
#include "kvc_prefill_tc.cuh"

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
    // one kernel per (element type, head width): the group only changes how
    // the CTA's 128 query rows map to (head, token)
    return G >= 1 && G <= TcPrefillCfg<KVC_ELEM, KVC_INST_D>::BM ? prefill_tc_info<KVC_ELEM, KVC_INST_D>() : nullptr;
}

}  // namespace kvc
