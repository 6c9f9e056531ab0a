// zc_decode_core.cuh -- decoding one chunk of a coded stream whose fixed part and escape section
// are staged in shared memory, by 128 threads.  Used by the decode kernel and by the loopback
// (compress and decompress in one launch), so the two decode with the same code.
//
// Method: ZipCCL (SIGCOMM scribe notes), "Key idea and contribution": in-window exponents are
// e0 + code, out-of-window exponents come from the separate store of full exponents (a list of
// (position, exponent) pairs, or a plane of every exponent when more than a third of the chunk
// escapes), so the reconstruction is exact (first technique).
//
// A thread holds 4 slices of 8 values; per slice it takes its 24 code bits and 8 sign|mantissa
// bytes from shared memory, builds two values per 32-bit word with a few integer ops, and writes
// one coalesced 16-byte store, escaped values with a placeholder exponent.  Then the threads walk
// a list together, one entry each, check it against the codes and patch the value, so escape
// work is proportional to the number of escapes rather than to the busiest lane.  A section of a
// plane's size is built from instead in the same single pass (sign|mantissa bytes plus the
// plane's exponents, each checked against its code), and again from the codes in the rare case
// that the count shows a list of that size.  Any disagreement with the canonical form sets
// ZC_ERR_CORRUPT.
#pragma once

#include "zc_common.cuh"

namespace zc {
namespace {

// A chunk whose escape section has the size of a plane: this thread's values built straight
// from the plane's exponents, each exponent checked against its value's code.  Returns this
// thread's code-7 count, with bit 31 set if an exponent disagrees with its code.  Kept out of
// line, off the path of chunks with a list.
__device__ __noinline__ unsigned plane_values(const uint8_t* codes, const uint8_t* smp, const uint8_t* plane,
                                              uint16_t* dst, unsigned m, int e0) {
  const unsigned tid = threadIdx.x & (kChunkThreads - 1);
  const bool full = m == kChunk;
  unsigned count = 0, bad = 0;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const unsigned g = 128 * q + tid, v0 = 8 * g;
    if (!full && v0 >= m) continue;
    const unsigned b = 3 * g;
    const uint32_t* cw = reinterpret_cast<const uint32_t*>(codes + (b & ~3u));
    const uint32_t bits = __funnelshift_r(cw[0], cw[1], 8 * (b & 3));
    const uint2 sm = *reinterpret_cast<const uint2*>(smp + v0);
    const uint2 ex = *reinterpret_cast<const uint2*>(plane + v0);
    uint32_t x[4];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const unsigned E = ((j < 4 ? ex.x : ex.y) >> (8 * (j & 3))) & 0xFFu;
      const unsigned s8 = ((j < 4 ? sm.x : sm.y) >> (8 * (j & 3))) & 0xFFu;
      const unsigned d = E - static_cast<unsigned>(e0);
      if ((full || v0 + j < m) && (d <= 6u ? d : 7u) != ((bits >> (3 * j)) & 7u)) bad = 1u;
      const uint32_t val = ((s8 & 0x80u) << 8) | (E << 7) | (s8 & 0x7Fu);
      x[j >> 1] = (j & 1) ? (x[j >> 1] | (val << 16)) : val;
    }
    uint32_t e = bits & (bits >> 1) & (bits >> 2) & 0x249249u;  // code 7: bit 3j for value j
    if (full || v0 + 8 <= m) {
      *reinterpret_cast<uint4*>(dst + v0) = make_uint4(x[0], x[1], x[2], x[3]);
    } else {
      e &= (1u << (3 * (m - v0))) - 1u;
      for (unsigned j = 0; v0 + j < m; ++j) dst[v0 + j] = static_cast<uint16_t>(pick4(x, j >> 1) >> (16 * (j & 1)));
    }
    count += __popc(e);
  }
  return count | (bad << 31);
}

// Decode chunk values [0, m) into dst.  fixed: the chunk's codes (code_section_bytes(m)) then its
// sign|mantissa plane; esc: its escape section (esc_bytes); both staged in shared memory and
// visible to every thread.  *escapes (shared) must be 0 on entry.  tid in [0, 128); bar() is a
// barrier over exactly those 128 threads.
template <typename Bar>
__device__ __forceinline__ void decode_chunk(const uint4* fixed, const uint4* esc, unsigned* escapes, uint16_t* dst,
                                             unsigned m, int e0, unsigned esc_bytes, int* status, unsigned tid,
                                             Bar bar) {
  const unsigned lane = tid & 31;
  const bool full = m == kChunk;
  const unsigned cbytes = full ? kFullCodeBytes : static_cast<unsigned>(code_section_bytes(m));
  const unsigned smbytes = full ? kChunk : static_cast<unsigned>(pad16(m));
  const uint8_t* codes = reinterpret_cast<const uint8_t*>(fixed);
  const uint8_t* smp = codes + cbytes;
  const uint8_t* esc_s = reinterpret_cast<const uint8_t*>(esc);
  const uint32_t e0_field = static_cast<uint32_t>(e0) * (128u * 0x00010001u);  // e0 << 7 in both halves

  // Every value as if in the window (an escape gets a placeholder exponent, patched below);
  // returns this thread's code-7 count.
  auto placeholders = [&]() -> unsigned {
    unsigned mine = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const unsigned g = 128 * q + tid, v0 = 8 * g;
      if (!full && v0 >= m) continue;
      const unsigned b = 3 * g;
      const uint32_t* cw = reinterpret_cast<const uint32_t*>(codes + (b & ~3u));
      const uint32_t bits = __funnelshift_r(cw[0], cw[1], 8 * (b & 3));
      const uint2 sm = *reinterpret_cast<const uint2*>(smp + v0);
      uint32_t x[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        // codes of values 2i, 2i+1 -> (c + e0) << 7 in the two halves
        const uint32_t v = (bits >> (6 * i)) & 0x3Fu;
        const uint32_t efield = (v & 0x38u) * (0x1FFFu << 7) + v * 128u + e0_field;
        // sign|mantissa bytes -> halves with the sign replicated over bits 7..15
        const uint32_t sw = i < 2 ? sm.x : sm.y;
        const unsigned lo = (2 * i) & 3;
        const uint32_t s2 = prmt(sw, 0u, lo | ((8u | lo) << 4) | ((lo + 1) << 8) | ((8u | (lo + 1)) << 12));
        x[i] = (s2 & 0x807F807Fu) | (efield & 0x7F807F80u);
      }
      uint32_t e = bits & (bits >> 1) & (bits >> 2) & 0x249249u;  // code 7: bit 3j for value j
      if (full || v0 + 8 <= m) {
        *reinterpret_cast<uint4*>(dst + v0) = make_uint4(x[0], x[1], x[2], x[3]);
      } else {
        e &= (1u << (3 * (m - v0))) - 1u;  // padding codes are checked below
        for (unsigned j = 0; v0 + j < m; ++j) dst[v0 + j] = static_cast<uint16_t>(pick4(x, j >> 1) >> (16 * (j & 1)));
      }
      mine += __popc(e);
    }
    return mine;
  };
  // A section of a plane's size (pad16(m) bytes) is a plane unless it is a list whose padded size
  // happens to match (3k within 15 bytes below m): build the values from it directly, and
  // again from the codes should the count below show a list.
  const bool plane_size = esc_bytes == pad16(m);
  bool plane_bad = false;
  unsigned mine;
  if (plane_size) {
    const unsigned r = plane_values(codes, smp, esc_s, dst, m, e0);
    mine = r & 0x7FFFFFFFu;
    plane_bad = (r >> 31) != 0;
  } else {
    mine = placeholders();
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mine += __shfl_xor_sync(0xFFFFFFFFu, mine, o);
  if (lane == 0) atomicAdd(escapes, mine);
  bar();  // every value is written and the chunk's escape count is known

  // Escapes.  k, the code-7 count, decides the section's form (a list when 3k <= m, else a
  // plane of every exponent) and so its size.  A list must name exactly the escaped values:
  // positions strictly increasing, below m, each holding code 7, each exponent outside the
  // window.  A plane must agree with the codes everywhere.  Either way the stream is canonical.
  const unsigned k = *reinterpret_cast<volatile unsigned*>(escapes);
  const bool plane = exponent_plane(m, k);
  bool corrupt = escape_section_bytes(m, k) != esc_bytes;
  if (!corrupt && plane) {
    corrupt = plane_bad;  // a plane always has a plane's size, so its values are in place
  } else if (!corrupt) {
    if (plane_size) {  // a list after all (the same in every thread): placeholders first
      placeholders();
      bar();
    }
    // A list: the threads walk it together, one entry each, check each entry against the codes
    // and the entry before it, and patch the value.
    auto patch = [&](unsigned i, unsigned pos, unsigned E, unsigned prev) {
      const unsigned pb = 3 * pos;
      const unsigned code = pos < m ? ((codes[pb >> 3] | (codes[(pb >> 3) + 1] << 8)) >> (pb & 7)) & 7u : 0u;
      if (code != 7u || (i > 0 && pos <= prev) ||
          (E >= static_cast<unsigned>(e0) && E <= static_cast<unsigned>(e0) + 6)) {
        corrupt = true;
        return;
      }
      const unsigned sm = smp[pos];
      dst[pos] = static_cast<uint16_t>(((sm & 0x80u) << 8) | (E << 7) | (sm & 0x7Fu));
    };
    const uint16_t* pos_list = reinterpret_cast<const uint16_t*>(esc_s);
    for (unsigned i = tid; i < k; i += kChunkThreads) patch(i, pos_list[i], esc_s[2 * k + i], i ? pos_list[i - 1] : 0u);
  }

  // zero padding: the escape section always, code bits and sign|mantissa bytes of a partial chunk
  const unsigned used = plane ? m : 3 * k;
  const unsigned epad = corrupt ? 0u : esc_bytes - used;  // < 16
  if (tid < epad) corrupt |= esc_s[used + tid] != 0;
  if (!full) {
    if (tid < smbytes - m) corrupt |= smp[m + tid] != 0;
    const unsigned bit = 3 * m + tid;  // at most 127 padding bits
    if (bit < 8 * cbytes) corrupt |= ((codes[bit >> 3] >> (bit & 7)) & 1u) != 0;
  }
  if (corrupt) set_error(status, ZC_ERR_CORRUPT);
}

}  // namespace
}  // namespace zc
