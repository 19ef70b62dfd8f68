// Kernel launches that report their own status.
//
// A <<< >>> launch returns nothing, and cudaGetLastError() after it returns,
// and clears, the last error of any earlier runtime call on the thread: an
// unrelated error the caller left pending would be reported as this launch's
// failure and lost to the caller.  cudaLaunchKernel returns the status of the
// launch itself (plus errors that already broke the context, which any call
// returns).  Every kernel of the library takes one parameter struct.
#pragma once

#include <cuda_runtime.h>

#include "dsv4kv.h"

namespace dsv4 {

template <typename P>
inline int launch_kernel(void (*kernel)(P), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                         const P &p)
{
    void *args[] = {const_cast<P *>(&p)};
    return cudaLaunchKernel(reinterpret_cast<const void *>(kernel), grid, block, args, smem,
                            stream) == cudaSuccess
               ? DSV4_OK
               : DSV4_ERR_CUDA;
}

}  // namespace dsv4
