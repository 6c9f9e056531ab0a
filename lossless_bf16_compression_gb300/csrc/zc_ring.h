// zc_ring.h -- where an escape section goes in an encoder CTA's ring buffer.  Pure arithmetic,
// shared by the encode kernel and a host-side check that replays random traces through it.
#pragma once

#if defined(__CUDACC__)
#define ZC_HOST_DEVICE __host__ __device__ __forceinline__
#else
#define ZC_HOST_DEVICE inline
#endif

namespace zc {

// The ring holds sections in the order they were placed; the ones still waiting end at offset
// `head`, contiguous modulo `ring_bytes`.  A section of `need` bytes goes at head when it fits
// before the end of the ring, else at offset 0 after the `gap` up to the end is skipped.  A
// section that ended exactly at the end leaves head = ring_bytes, which is offset 0.  The place
// depends on head alone, so every thread that tracks the same head takes the same decision.
ZC_HOST_DEVICE void ring_place(unsigned head, unsigned need, unsigned ring_bytes, unsigned* where, unsigned* gap) {
  const unsigned h = head >= ring_bytes ? 0u : head;
  const unsigned g = (need && h + need > ring_bytes) ? ring_bytes - h : 0u;
  *where = g ? 0u : h;
  *gap = g;
}

// Whether the section fits now: the bytes still waiting (gaps included), the gap and the section
// itself within the ring.  A drained ring takes any section of up to ring_bytes / 2 bytes (the gap
// is shorter than the section).
ZC_HOST_DEVICE bool ring_fits(unsigned waiting, unsigned gap, unsigned need, unsigned ring_bytes) {
  return waiting + gap + need <= ring_bytes;
}

}  // namespace zc
