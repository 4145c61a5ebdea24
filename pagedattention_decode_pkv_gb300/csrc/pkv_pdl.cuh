// Programmatic dependent launch (PDL) helpers shared by the library's kernels.
//
// Every kernel is launched with programmatic stream serialization allowed, so
// the next kernel in the stream can be scheduled while the previous one
// drains.  Each kernel therefore executes pdl_wait() before its first access
// to global memory (read or write): the wait returns once the preceding grid
// has completed and its writes are visible, so no data hazard is possible.
// pdl_trigger() lets the dependent grid start launching; it is issued right
// after the wait, when every CTA of the current grid is already resident or
// has been scheduled.
#pragma once

#include <cuda_runtime.h>

namespace pkv {

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Which launches allow programmatic dependent launch (the kernels always
// execute pdl_wait(), which is a no-op without it).  Measured on GB300 over a
// whole decode step (slot mapping, store, attention + combine, unpack K/V):
// chaining everything but the unpack is fastest; letting the many-wave unpack
// grid start early as well cost ~9 % of the step.
constexpr bool kPdlSlotMapping = true;
constexpr bool kPdlStore = true;
constexpr bool kPdlDecode = true;
constexpr bool kPdlCombine = true;
constexpr bool kPdlUnpack = false;

// Launch `kernel` on `stream`, with programmatic stream serialization allowed
// when `pdl` is set.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(bool pdl, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

}  // namespace pkv
