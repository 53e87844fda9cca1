// A named NVTX range over one C-ABI call, so that a profiler's timeline shows
// which call launched which kernels (and ncu --nvtx can select by call). The
// range covers the host side of the call: validation and launches, the calls
// being asynchronous. NVTX v3 is header-only; without a profiler attached a push
// or pop returns at once.
#pragma once

#if __has_include(<nvtx3/nvToolsExt.h>)
#include <nvtx3/nvToolsExt.h>
#define PA_HAVE_NVTX 1
#else
#define PA_HAVE_NVTX 0     // a toolkit without the NVTX headers: the ranges compile to nothing
#endif

namespace pa {

struct CallRange {
#if PA_HAVE_NVTX
    explicit CallRange(const char *name) { nvtxRangePushA(name); }
    ~CallRange() { nvtxRangePop(); }
#else
    explicit CallRange(const char *) {}
#endif
    CallRange(const CallRange &) = delete;
    CallRange &operator=(const CallRange &) = delete;
};

}  // namespace pa
