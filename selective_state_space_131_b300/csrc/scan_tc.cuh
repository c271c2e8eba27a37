// scan_tc.cuh -- chunked tensor-core (tcgen05) prefill.  (placeholder)
#pragma once
#include "m3scan.h"
namespace m3tc {
inline bool supports(const m3_dims&) { return false; }
inline int launch(const m3_dims&, const void*, const float*, const float*, const void*, const void*, const float*,
                  const void*, void*, float*, cudaStream_t) {
    return M3_ERR_UNSUPPORTED;
}
}  // namespace m3tc
