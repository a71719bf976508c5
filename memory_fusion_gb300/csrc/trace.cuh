// trace.cuh -- optional %globaltimer timeline stamps of the persistent
// kernels: per CTA, slots 0..3 (start, set-up done, role loops done, exit),
// then CF_TRACE_EVENTS slots for each of the CTA's first CF_TRACE_TILES
// tiles.  A null buffer disables tracing (one predictable branch per stamp).
#pragma once

#include "../../include/cf.h"
#include "ptx.cuh"

namespace cf {

__device__ __forceinline__ void trace_stamp(unsigned long long *tr, int slot) {
    if (tr != nullptr) tr[blockIdx.x * CF_TRACE_SLOTS + slot] = ptx::globaltimer();
}
__device__ __forceinline__ void trace_tile(unsigned long long *tr, int tile, int ev) {
    if (tr != nullptr && tile < CF_TRACE_TILES)
        tr[blockIdx.x * CF_TRACE_SLOTS + 4 + tile * CF_TRACE_EVENTS + ev] = ptx::globaltimer();
}
__device__ __forceinline__ void trace_tile_value(unsigned long long *tr, int tile, int ev, unsigned long long v) {
    if (tr != nullptr && tile < CF_TRACE_TILES) tr[blockIdx.x * CF_TRACE_SLOTS + 4 + tile * CF_TRACE_EVENTS + ev] = v;
}

}  // namespace cf
