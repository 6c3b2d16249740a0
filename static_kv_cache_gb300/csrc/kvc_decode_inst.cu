// kvc_decode_inst.cu -- explicit decode kernels for one (element type, head
// width), selected at compile time by KVC_INST_TYPE (0 bf16, 1 fp16, 2 fp32)
// and KVC_INST_D.  The build compiles this file once per pair, in parallel.
#include "kvc_decode_mma.cuh"
#if defined(KVC_INST_TC)
#include "kvc_decode_tc.cuh"
#endif

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
#define KVC_ELEM float
#define KVC_TAG f32
#endif

#define KVC_CAT2(a, b, c) decode_kernel_##a##_##b
#define KVC_CAT(a, b) KVC_CAT2(a, b, 0)
#define KVC_TABLE_FN KVC_CAT(KVC_TAG, KVC_INST_D)

namespace kvc {

// 16-bit caches with 2 to 8 query heads per KV head and d_h of 64 or 128 run
// the tensor-core kernel; one query head per KV head, fp32 caches and the
// other head widths run the CUDA-core kernel.  Groups of 16, 32 and 64 heads
// (multi-query attention) run the tensor-core kernel only.
#if KVC_INST_TYPE != 2 && (KVC_INST_D == 64 || KVC_INST_D == 128)
#define KVC_GROUPED(G) mma_decode_info<KVC_ELEM, KVC_INST_D, G>()
#define KVC_LARGE_GROUP(G) mma_decode_info<KVC_ELEM, KVC_INST_D, G>()
#else
#define KVC_GROUPED(G) decode_info<KVC_ELEM, KVC_INST_D, G>()
#define KVC_LARGE_GROUP(G) nullptr
#endif

#if defined(KVC_INST_TC)
// The tcgen05 kernel of 16- and 32-head groups at d_h = 128 (contiguous
// caches bound to a handle); the build compiles this variant once per 16-bit
// type.
#if KVC_INST_D != 128 || KVC_INST_TYPE == 2
#error "the tcgen05 decode variant is built for 16-bit caches with d_h = 128"
#endif
#define KVC_TCAT2(a) decode_kernel_tc_##a##_128
#define KVC_TCAT(a) KVC_TCAT2(a)
const DecodeKernelInfo *KVC_TCAT(KVC_TAG)(int G) {
    switch (G) {
        case 16: return tc_decode_info<KVC_ELEM, 16>();
        case 32: return tc_decode_info<KVC_ELEM, 32>();
        default: return nullptr;
    }
}
#elif defined(KVC_INST_PAGED)
// Kernels for paged pools, built once per 16-bit type and d_h of 64 or 128:
// the kernels that read a block two KV heads at a time (2 or 4 query heads
// per KV head; G2 counts the query heads of both), and for d_h = 128 the
// kernels that read one KV head per block in the half-row tile layout.
#if (KVC_INST_D != 128 && KVC_INST_D != 64) || KVC_INST_TYPE == 2
#error "the paged variant is built for 16-bit caches with d_h = 64 or 128"
#endif
#define KVC_PAIR2(a, d) decode_kernel_pair_##a##_##d
#define KVC_PAIR(a, d) KVC_PAIR2(a, d)
const DecodeKernelInfo *KVC_PAIR(KVC_TAG, KVC_INST_D)(int G2) {
    switch (G2) {
        case 4: return mma_decode_info<KVC_ELEM, KVC_INST_D, 4, true, true>();
        case 8: return mma_decode_info<KVC_ELEM, KVC_INST_D, 8, true, true>();
        default: return nullptr;
    }
}
#if KVC_INST_D == 128
#define KVC_PCAT2(a) decode_kernel_paged_##a##_128
#define KVC_PCAT(a) KVC_PCAT2(a)
const DecodeKernelInfo *KVC_PCAT(KVC_TAG)(int G) {
    switch (G) {
        case 2: return mma_decode_info<KVC_ELEM, 128, 2, true>();
        case 3: return mma_decode_info<KVC_ELEM, 128, 3, true>();
        case 4: return mma_decode_info<KVC_ELEM, 128, 4, true>();
        case 5: return mma_decode_info<KVC_ELEM, 128, 5, true>();
        case 6: return mma_decode_info<KVC_ELEM, 128, 6, true>();
        case 7: return mma_decode_info<KVC_ELEM, 128, 7, true>();
        case 8: return mma_decode_info<KVC_ELEM, 128, 8, true>();
        case 16: return mma_decode_info<KVC_ELEM, 128, 16, true>();
        case 32: return mma_decode_info<KVC_ELEM, 128, 32, true>();
        case 64: return mma_decode_info<KVC_ELEM, 128, 64, true>();
        default: return nullptr;
    }
}
#endif
#else
const DecodeKernelInfo *KVC_TABLE_FN(int G) {
    switch (G) {
        case 1: return decode_info<KVC_ELEM, KVC_INST_D, 1>();
        case 2: return KVC_GROUPED(2);
        case 3: return KVC_GROUPED(3);
        case 4: return KVC_GROUPED(4);
        case 5: return KVC_GROUPED(5);
        case 6: return KVC_GROUPED(6);
        case 7: return KVC_GROUPED(7);
        case 8: return KVC_GROUPED(8);
        case 16: return KVC_LARGE_GROUP(16);
        case 32: return KVC_LARGE_GROUP(32);
        case 64: return KVC_LARGE_GROUP(64);
        default: return nullptr;
    }
}
#endif

}  // namespace kvc
