// Search kernels over partial induced subgraphs of second-level subtrees, one per row width.
#define MCE_SEARCH_IP 1
#define MCE_SEARCH_L2 1
#include "search_impl.cuh"

namespace mce {

const void *search_kernel_partial_l2(int cls)
{
    switch (cls) {
    case 0: return (const void *)search_kernel<1>;
    case 1: return (const void *)search_kernel<2>;
    case 2: return (const void *)search_kernel<4>;
    case 3: return (const void *)search_kernel<8>;
    case 4: return (const void *)search_kernel<16>;
    default: return (const void *)search_kernel<32>;
    }
}

}  // namespace mce
