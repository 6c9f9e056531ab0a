// zc_code_core.cuh -- coding of one thread's 32 consecutive values of a chunk (3-bit codes,
// sign|mantissa bytes, escape flags), the stores of its share of the chunk's fixed part, and the
// writing of its escapes into a chunk's list.  Shared by the persistent encoder and the
// small-tensor kernel, so both code with the same instructions.
//
// Method: ZipCCL (SIGCOMM scribe notes), "Key idea and contribution", first technique: an
// exponent inside the window [e0, e0 + 6] becomes a 3-bit code, any other one is an escape (code
// 7) kept whole in the chunk's separate store; sign and mantissa are kept as they are.
#pragma once

#include "zc_common.cuh"

namespace zc {
namespace {

// The 8 code-7 flags of a slice (bit 3j for value j) as bits 0..7.
__device__ __forceinline__ unsigned compact8(unsigned m) {
  m = (m | (m >> 2)) & 0x0C30C3u;
  m = (m | (m >> 4)) & 0x00F00Fu;
  return (m | (m >> 8)) & 0xFFu;
}

// Index of the highest set bit of a nonzero word.
__device__ __forceinline__ unsigned msb_index(unsigned x) {
  unsigned b;
  asm("bfind.u32 %0, %1;" : "=r"(b) : "r"(x));
  return b;
}

// A thread's 32 consecutive values v0 .. v0 + 31, coded.
struct Coded32 {
  uint32_t g[4];   // 24-bit code groups: code j of group q at bits [3j, 3j + 3)
  uint32_t sm[8];  // sign|mantissa bytes, four per word
  uint32_t e[4];   // code-7 flags: bit 3j of e[q] for value v0 + 8q + j
};

// xv[q] holds values v0 + 8q .. v0 + 8q + 7.  Values at or past m (a ragged chunk, full == false)
// get code 0, byte 0 and no escape.  kadd = ((256 - e0) << 7) in both halves (codes7_x2).
__device__ __forceinline__ void code32(const uint4 (&xv)[4], uint32_t kadd, unsigned v0, unsigned m, bool full,
                                       Coded32& k) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t w[4] = {xv[q].x, xv[q].y, xv[q].z, xv[q].w};
    uint32_t c7[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) c7[i] = codes7_x2(w[i], kadd);
    if (!full) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const unsigned v = v0 + 8 * q + 2 * i;
        const uint32_t keep = (v < m ? 0x0000FFFFu : 0u) | (v + 1 < m ? 0xFFFF0000u : 0u);
        c7[i] &= keep;
        w[i] &= keep;
      }
    }
    k.sm[2 * q] = sign_mantissa_x4(w[0], w[1]);
    k.sm[2 * q + 1] = sign_mantissa_x4(w[2], w[3]);
    k.g[q] = pack_codes8(c7);
    k.e[q] = k.g[q] & (k.g[q] >> 1) & (k.g[q] >> 2) & 0x249249u;  // code 7
  }
}

// The thread's share of the chunk's fixed part at `fixed` (global or generic address): its 12
// code bytes at 3 v0 / 8 of the code section (cbytes long) and its 32 sign|mantissa bytes at v0
// of the plane (smbytes long, after the codes); nothing past the sections of a ragged chunk.
__device__ __forceinline__ void store_fixed32(uint8_t* fixed, unsigned cbytes, unsigned smbytes, unsigned v0,
                                              bool full, const Coded32& k) {
  uint8_t* const smp = fixed + cbytes + v0;
  if (full || v0 < smbytes) *reinterpret_cast<uint4*>(smp) = make_uint4(k.sm[0], k.sm[1], k.sm[2], k.sm[3]);
  if (full || v0 + 16 < smbytes) *reinterpret_cast<uint4*>(smp + 16) = make_uint4(k.sm[4], k.sm[5], k.sm[6], k.sm[7]);
  const uint32_t cw[3] = {k.g[0] | (k.g[1] << 24), (k.g[1] >> 8) | (k.g[2] << 16), (k.g[2] >> 16) | (k.g[3] << 8)};
  uint32_t* const cp = reinterpret_cast<uint32_t*>(fixed + 3 * v0 / 8);
#pragma unroll
  for (int i = 0; i < 3; ++i)
    if (full || 3 * v0 / 8 + 4 * i < cbytes) cp[i] = cw[i];
}

// The thread's escapes into a chunk's list at `esc` (shared-window address of the section; k
// escapes in the chunk, this thread's first rank `base`, its flags m32 with value v0 + b at bit
// b, cnt of them): u16 positions at esc + 2 rank, u8 exponents at esc + 2k + rank.  exp_at(b)
// returns value v0 + b's exponent.  `dense` (some lane of the warp holds 16 or more escapes):
// lane L takes its escapes from value L - 1 downwards (mod 32), so that the lanes' stores and
// loads, 32 ranks apart in the plain order, fall in different banks.
template <typename ExpAt>
__device__ __forceinline__ void write_list32(unsigned m32, unsigned cnt, unsigned v0, unsigned base, unsigned k,
                                             uint32_t esc, bool dense, ExpAt exp_at) {
  if (!dense) {
    // highest value first: ranks base + cnt - 1 down to base
    uint32_t at16 = esc + 2 * (base + cnt), at8 = esc + 2 * k + base + cnt;  // one past the last
    unsigned mm = m32;
    while (mm) {
      const unsigned b = msb_index(mm);
      mm ^= 1u << b;
      at16 -= 2;
      at8 -= 1;
      sts_u16(at16, v0 + b);
      sts_u8(at8, exp_at(b));
    }
  } else {
    const unsigned rot = threadIdx.x & 31;
    unsigned mm = __funnelshift_r(m32, m32, rot);  // value b at bit (b - rot) mod 32
    while (mm) {
      const unsigned bp = msb_index(mm);
      mm ^= 1u << bp;
      const unsigned b = (bp + rot) & 31;
      const unsigned r = base + __popc(m32 & ((1u << b) - 1u));
      sts_u16(esc + 2 * r, v0 + b);
      sts_u8(esc + 2 * k + r, exp_at(b));
    }
  }
}

}  // namespace
}  // namespace zc
