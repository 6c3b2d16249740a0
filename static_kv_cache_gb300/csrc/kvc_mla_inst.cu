// kvc_mla_inst.cu -- the MLA decode kernels for one 16-bit element type,
// selected at compile time by KVC_INST_TYPE (0 bf16, 1 fp16): latent widths
// d_c of 128, 256 and 512 with 8 or 16 query heads.
#include "kvc_mla.cuh"

#ifndef KVC_INST_TYPE
#error "KVC_INST_TYPE must be defined"
#endif

#if KVC_INST_TYPE == 0
#define KVC_ELEM __nv_bfloat16
#define KVC_MLA_TABLE mla_kernel_bf16
#elif KVC_INST_TYPE == 1
#define KVC_ELEM __half
#define KVC_MLA_TABLE mla_kernel_f16
#else
#error "the MLA kernels take 16-bit caches"
#endif

namespace kvc {

const MlaKernelInfo *KVC_MLA_TABLE(int d_c, int H) {
    if (H == 8) {
        if (d_c == 128) return mla_info<KVC_ELEM, 128, 8>();
        if (d_c == 256) return mla_info<KVC_ELEM, 256, 8>();
        if (d_c == 512) return mla_info<KVC_ELEM, 512, 8>();
    } else if (H == 16) {
        if (d_c == 128) return mla_info<KVC_ELEM, 128, 16>();
        if (d_c == 256) return mla_info<KVC_ELEM, 256, 16>();
        if (d_c == 512) return mla_info<KVC_ELEM, 512, 16>();
    }
    return nullptr;
}

}  // namespace kvc
