// Programmatic dependent launch for the short kernels of a step: the token
// append and the decode-set upload ahead of the decode kernel, and block
// mass, scoring, selection, gather plan and mirror copy after it.
//
// A kernel launched with launch_pdl() may be scheduled while the kernel
// before it in the stream is still running: its CTAs start, do what depends
// on nothing that kernel writes, and block in pdl_wait() until that kernel
// has completed and its memory is visible.  This hides the launch and ramp
// of each short kernel behind the tail of the previous one.  Rules every
// kernel launched this way follows:
//   - every thread calls pdl_wait() before it reads or writes memory that an
//     earlier kernel of the stream may still write, and before it exits (so
//     that the grid completes only after its predecessor has, which keeps
//     the ordering transitive along the chain);
//   - before pdl_wait() it reads only data that was final before the last
//     normally-launched kernel ahead of it started: the decode set and the
//     block records, final before the decode kernel (a normal launch) starts.
//     The set upload and the token append are launched this way too, but
//     touch memory only after their own pdl_wait(), and a normally-launched
//     kernel (the decode kernel, or the mass copy of a debug set) follows
//     every set upload before anything reads the set.
// The decode kernels trigger their dependents at their start, so that the
// combine kernel's CTAs are in place when the decode completes.
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
