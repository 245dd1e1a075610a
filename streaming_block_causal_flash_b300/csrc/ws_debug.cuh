// ws_debug.cuh -- bounds checks of the debug build (compiled with -DWS_DEBUG=1
// into libws_b300_debug.so; selected at run time by WS_DEBUG=1).
//
// WS_BOUND(word, idx, limit, site) guards one global-memory access whose index
// the kernel computed: it is true when 0 <= idx < limit.  Otherwise it records
// code 3 and (site << 16) | (block index & 0xFFFF) in the translation unit's
// device error word (the first failure wins) and is false, so that the guarded
// access is skipped: a bad index never reaches memory, nothing traps.  In the
// normal build the macro is the constant true and costs nothing.
//
// Check sites (reported by ws_get_device_error): 21 attention output row,
// 22 attention LSE, 23 split-KV partial write, 24 merge read of a partial,
// 25 merge output row, 26 merge LSE, 31 append source, 32 append cache row
// (27 and 28 are no longer used).  The Euler kernels index by their loop
// counters alone, whose loop bounds are the checks; TMA copies (the fused
// commit's stores, the append's tensor store) are clipped by their tensor
// maps, whose extents end at the rows they may write.
#pragma once

#ifndef WS_DEBUG
#define WS_DEBUG 0
#endif

namespace ws {

__device__ __forceinline__ bool bound_fail(unsigned int* word, int site) {
  if (atomicCAS(&word[0], 0u, 3u) == 0u)
    word[1] = (static_cast<unsigned>(site) << 16) | (blockIdx.x & 0xFFFFu);
  return false;
}

}  // namespace ws

#if WS_DEBUG
#define WS_BOUND(word, idx, limit, site)                                          \
  ((static_cast<unsigned long long>(static_cast<long long>(idx)) <                \
    static_cast<unsigned long long>(static_cast<long long>(limit))) ||            \
   ::ws::bound_fail((word), (site)))
#else
#define WS_BOUND(word, idx, limit, site) true
#endif
