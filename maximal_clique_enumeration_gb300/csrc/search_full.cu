// Search kernels over full induced subgraphs of first-level subtrees, one per row width and
// launch group.
#define MCE_SEARCH_IP 0
#define MCE_SEARCH_L2 0
#include "search_impl.cuh"

namespace mce {

const void *search_kernel_full(int cls, bool big)
{
    switch (cls) {
    case 0: return big ? (const void *)search_kernel<1, true> : (const void *)search_kernel<1, false>;
    case 1: return big ? (const void *)search_kernel<2, true> : (const void *)search_kernel<2, false>;
    case 2: return big ? (const void *)search_kernel<4, true> : (const void *)search_kernel<4, false>;
    case 3: return big ? (const void *)search_kernel<8, true> : (const void *)search_kernel<8, false>;
    case 4: return big ? (const void *)search_kernel<16, true> : (const void *)search_kernel<16, false>;
    default: return big ? (const void *)search_kernel<32, true> : (const void *)search_kernel<32, false>;
    }
}

const void *search_kernel_full_rec(int cls, bool big)
{
    switch (cls) {
    case 0: return big ? (const void *)search_kernel<1, true, true> : (const void *)search_kernel<1, false, true>;
    case 1: return big ? (const void *)search_kernel<2, true, true> : (const void *)search_kernel<2, false, true>;
    default: return big ? (const void *)search_kernel<4, true, true> : (const void *)search_kernel<4, false, true>;
    }
}

const void *build_kernel_full(int cls)
{
    switch (cls) {
    case 0: return (const void *)build_kernel<1>;
    case 1: return (const void *)build_kernel<2>;
    default: return (const void *)build_kernel<4>;
    }
}

}  // namespace mce
