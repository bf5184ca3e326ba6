// Programmatic dependent launch for the kernels of a step: the token append,
// the decode-set upload, the decode kernels, and block mass, scoring,
// selection, gather plan and mirror copy after them.
//
// A kernel launched with launch_pdl() may be scheduled while the kernel
// before it in the stream is still running: its CTAs start, do what depends
// on nothing that kernel writes, and block in pdl_wait() until that kernel
// has completed and its memory is visible.  This hides the launch and ramp
// of each kernel behind the tail of the previous one.  Rules every kernel
// launched this way follows:
//   - every thread calls pdl_wait() before it reads or writes memory that an
//     earlier kernel of the stream may still write, and before it exits (so
//     that the grid completes only after its predecessor has, which keeps
//     the ordering transitive along the chain);
//   - a kernel triggers its dependents (pdl_trigger) only after its own
//     pdl_wait() has returned, so that when a kernel starts, every kernel two
//     or more launches ahead of it has completed.  The one exception is the
//     set upload, which triggers at its start; the kernel after it (a decode
//     kernel, or a plain launch) touches no memory before its own wait;
//   - before pdl_wait() a kernel reads only data written two or more launches
//     ahead of it: the decode set and the block records, read early by the
//     combine, mass and selection kernels, are written by the set upload, the
//     token append, the scoring of earlier steps and plain launches (record
//     patches), never by the decode kernels or the kernels after them.
// The decode kernels trigger right after their wait, so that the combine
// kernel's CTAs are in place when the decode completes.
// After a copy or an event in the stream the attribute has no effect: the
// kernel starts after everything before it, as a plain launch would.
#pragma once

#include <utility>

#include <cuda_runtime.h>

namespace kvs {

__device__ __forceinline__ void pdl_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Lets the next kernel of the stream (if launched with launch_pdl) start its
// CTAs once every CTA of this grid has passed this point or exited.
__device__ __forceinline__ void pdl_trigger()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... Params, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t s, Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace kvs
