// chain.cuh -- programmatic dependent launch for the kernel chains of the
// batched decode step (one CUDA graph per step, 113 short kernels in stream
// order; every kernel after the first is chained) and of the prompt prefill
// (one graph, 112 kernels; only its GEMMs are chained, the rest measured
// slower chained).
//
// A kernel launched with the programmatic-serialization attribute may be
// scheduled while the kernel before it in the stream is still running: its
// CTAs become resident and wait in griddepcontrol.wait until that kernel
// has completed and its memory writes are visible.  This hides the launch
// and CTA-rasterisation latency of each link of the chain.  The rules that
// keep the chain's stream-order semantics:
//   * every kernel of a chain calls chain_enter() before its first access
//     to global memory (read or write), with all its threads; the only
//     work before it is on shared and tensor memory;
//   * chain_enter() releases the next kernel only after the wait, so at
//     most two kernels of the chain are resident at a time, and a kernel
//     completes only after its predecessor did (which makes the ordering
//     transitive: a kernel also sees the writes of every earlier kernel).
//     A chain may mix chained and plain launches: a plain launch waits for
//     its predecessor's completion as usual, which keeps the same order.
// Without the attribute (the first kernel of a chain, or GPT2_PDL=0 in the
// environment) both instructions are no-ops and the launches are plain
// stream-ordered launches.
#pragma once
#include <cuda_runtime.h>

#include <cstdlib>
#include <cstring>
#include <utility>

namespace gpt2 {

__device__ __forceinline__ void chain_enter() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Programmatic launches are on unless GPT2_PDL=0 (read once per process).
inline bool chain_pdl_enabled() {
    static const bool on = [] {
        const char* v = getenv("GPT2_PDL");
        return !(v && strcmp(v, "0") == 0);
    }();
    return on;
}

// kernel<<<grid, block, smem, st>>>(args...), with the programmatic-
// serialization attribute when `follows` (the launch follows another
// kernel of the same chain in stream order) and programmatic launches are on.
template <typename... KArgs, typename... Args>
cudaError_t chain_launch(bool follows, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                         cudaStream_t st, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    const bool pdl = follows && chain_pdl_enabled();
    cfg.attrs = pdl ? at : nullptr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace gpt2
