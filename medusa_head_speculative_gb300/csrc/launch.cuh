// Kernel launches with programmatic dependent launch (PDL).
//
// Every kernel of the library calls pdl_trigger() early (kernels that use TMEM right after
// allocating it), which lets the next kernel on the stream begin as soon as all of this
// kernel's CTAs have got that far, and calls pdl_wait()
// before it reads anything an earlier kernel wrote (griddepcontrol.wait returns once every
// earlier kernel on the stream has completed and its writes are visible).  What a kernel
// does before pdl_wait() touches only inputs that no kernel of the current call writes:
// weights, plan tables, the cached prefix K/V, and its own shared memory and TMEM.
//
// The first kernel of each public entry point is launched without the attribute, so it
// waits, as usual, for everything the caller queued before the call.
#pragma once
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <cstring>
#include <utility>

namespace medusa {

// True when the launch about to be made may overlap the previous one (an earlier kernel of
// the same entry point on the same stream); records this launch for the next call.
bool pdl_take(cudaStream_t st);
// Called on entry to every public function that launches kernels.
void pdl_reset();
// Kernels launched so far by the calling host thread.
long kernels_launched();

// Scope of one public entry point: the first launch inside it does not overlap earlier
// work, and the call shows up as an NVTX range (named after the entry point) in profilers.
struct EntryScope {
  explicit EntryScope(const char* name) {
    pdl_reset();
    nvtxRangePushA(name);
  }
  ~EntryScope() { nvtxRangePop(); }
  EntryScope(const EntryScope&) = delete;
  EntryScope& operator=(const EntryScope&) = delete;
};

template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                          int cluster_y, Args&&... args) {
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  std::memset(attr, 0, sizeof(attr));
  int n = 0;
  if (pdl_take(st)) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cluster_y > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = 1;
    attr[n].val.clusterDim.y = (unsigned)cluster_y;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = (unsigned)n;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

}  // namespace medusa
