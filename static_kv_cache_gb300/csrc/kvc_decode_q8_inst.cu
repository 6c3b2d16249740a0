// kvc_decode_q8_inst.cu -- decode kernels for int8 caches with one fp32
// scale per row (d_h = 128), one per query-group size.
#include "kvc_decode_q8.cuh"

namespace kvc {

const DecodeKernelInfo *decode_kernel_q8_128(int G) {
    switch (G) {
        case 1: return q8_decode_info<128, 1>();
        case 2: return q8_decode_info<128, 2>();
        case 3: return q8_decode_info<128, 3>();
        case 4: return q8_decode_info<128, 4>();
        case 5: return q8_decode_info<128, 5>();
        case 6: return q8_decode_info<128, 6>();
        case 7: return q8_decode_info<128, 7>();
        case 8: return q8_decode_info<128, 8>();
        default: return nullptr;
    }
}

}  // namespace kvc
