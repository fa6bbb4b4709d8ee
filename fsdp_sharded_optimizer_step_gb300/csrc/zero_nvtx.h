// NVTX ranges around the C-ABI calls: every call that queues device work (or
// runs the offloaded host update) opens a range named after itself, so a
// timeline tool (Nsight Systems, Nsight Compute's --nvtx filters) shows which
// call launched which kernels.  NVTX v3 is header-only; with no tool attached a
// range costs a few nanoseconds.  Not part of the C ABI.
#pragma once

#include <nvtx3/nvToolsExt.h>

namespace zero {

class NvtxRange {
  public:
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange &) = delete;
    NvtxRange &operator=(const NvtxRange &) = delete;
};

}  // namespace zero

// Opens a range named after the enclosing function until it returns.
#define ZERO_NVTX_RANGE() ::zero::NvtxRange zero_nvtx_range_(__func__)
