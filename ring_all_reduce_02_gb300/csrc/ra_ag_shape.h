// Launch shape of the all-gather kernel (build-time overridable for tuning
// sweeps): one compact read and N vector stores per element.
#pragma once

#include "ra_kernels.cuh"

#ifndef RA_AG_THREADS
#define RA_AG_THREADS 256
#endif
#ifndef RA_AG_MIN_BLOCKS
#define RA_AG_MIN_BLOCKS 2
#endif
#ifndef RA_AG_UNROLL
#define RA_AG_UNROLL 1
#endif

namespace ra {
using AgShape = Shape<RA_AG_THREADS, RA_AG_MIN_BLOCKS, RA_AG_UNROLL, 1>;
}  // namespace ra
