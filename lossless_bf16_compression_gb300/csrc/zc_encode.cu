// zc_encode.cu -- chunked encoder: 3-bit exponent codes, sign|mantissa byte plane, escape
// compaction, and a single-pass device-wide scan that places every escape list in one
// contiguous stream behind a chunk-offset table.
//
// Method: ZipCCL (SIGCOMM scribe notes), "Key idea and contribution": in-window exponents are
// coded in 3 bits, out-of-window exponents are kept whole in a list of their own (first
// technique); the kernels lay data out for the communication step, align their global and
// shared memory accesses, and overlap data movement with the coding (second technique).
//
// GB300 design.  A persistent grid, five CTAs per SM.  The first CTA to start is the scanner;
// every other CTA has four coding warps and one retiring warp, so that each chunk's fixed costs (waits,
// ranks, barriers) are paid by 128 threads and five chunks are in flight per SM (measured
// faster than eight coding warps at four CTAs per SM).  Chunks are handed out by an atomic
// ticket (ticket order = chunk order).  Inputs (8 KiB per chunk) arrive by tiled async copies
// (TMA engine, one box of a tensor map per chunk, mbarrier completion) into two stages, so the
// next chunk's copy is in flight while a chunk is coded (deeper pipelines measured slower:
// every stage holds a ticket, and held tickets lengthen the tail).  A coding thread holds 32
// consecutive values and codes two values per 32-bit word with packed 16-bit arithmetic; the
// copies use the 128-byte swizzle, so its four 16-byte reads of its own 64 bytes are free of
// bank conflicts.  The fixed part of a chunk has a place that follows from n, so it goes
// straight from registers to HBM: per thread two 16-byte stores of sign|mantissa bytes and
// three 32-bit words of codes.  Holding consecutive values makes a thread's escapes
// consecutive in the list, so each thread writes its own with one bit scan, two stores and one
// load per escape.  Only the escape list waits for the device-wide scan: each chunk publishes
// its list size in a per-chunk state word as soon as its escape count is known, and the
// scanner's four warps walk the state words in order, 1024 per round trip, turning every run
// of published sizes into inclusive offsets (a chained scan with one scanning block, after
// Merrill & Garland's single-pass scan).  Escape lists wait in a ring buffer in shared memory,
// where a waiting list costs only its own bytes; the retiring warp polls up to 32 waiting lists
// per round trip and copies resolved ones out with 16-byte stores, so coding never waits for
// the scan unless the ring is full.  Every wait is bounded.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "zc_code_core.cuh"
#include "zc_common.cuh"
#include "zc_decode_core.cuh"
#include "zc_ring.h"
#include "zc_stats_core.cuh"

namespace zc {
namespace {

constexpr int kCoders = 128;               // coding threads, 32 values each
static_assert(32 * kCoders == kChunk, "a coding thread holds 32 consecutive values");
constexpr int kThreads = kCoders + 32;     // + the retiring warp (idle in the scanning CTA)
#ifndef ZC_ENCODE_CTAS_PER_SM
#define ZC_ENCODE_CTAS_PER_SM 5
#endif
#ifndef ZC_ENCODE_RING_KB
#define ZC_ENCODE_RING_KB 18
#endif
#ifndef ZC_ENCODE_PREFETCH
#define ZC_ENCODE_PREFETCH 1
#endif
constexpr int kCtasPerSm = ZC_ENCODE_CTAS_PER_SM;
constexpr int kStages = 2;                 // input chunks in flight per CTA
constexpr unsigned kInBytes = 2 * kChunk;
// Escape-section ring per CTA: four and a half of the largest (a 4 KB plane).  Measured against
// 16, 20 and 24 KB: up to 18 KB the five CTAs' shared memory fits a smaller carveout, and the
// low-escape tensors coded about 4% faster than with 20 or 24 KB; 18 KB keeps that and gives the
// escape-heavy tensors, where the ring fills, 2% more than 16 KB.
constexpr unsigned kRingBytes = ZC_ENCODE_RING_KB * 1024;
static_assert(kRingBytes >= 2 * kMaxEscapeBytes, "a section placed after a skipped gap always fits a drained ring");
static_assert(kRingBytes % 16 == 0, "sections and their places are 16-byte aligned");
constexpr unsigned kQueue = 64;            // escape sections waiting, at most
constexpr unsigned kDenseMin = 16;         // escapes per lane from which a warp takes the dense loop
constexpr unsigned kWaitLimit = 1u << 22;  // mbarrier polls before giving up
constexpr int kScanPerLane = 8;            // state words per scanner lane per round trip
#ifndef ZC_LOOPBACK_CYCLE
#define ZC_LOOPBACK_CYCLE 5
#endif
#ifndef ZC_LOOPBACK_DECODERS
#define ZC_LOOPBACK_DECODERS 1
#endif
constexpr unsigned kLoopbackCycle = ZC_LOOPBACK_CYCLE;      // loopback: of every kLoopbackCycle CTAs (by
constexpr unsigned kLoopbackDecoders = ZC_LOOPBACK_DECODERS;  // start order), this many only decode
static_assert(kLoopbackDecoders < kLoopbackCycle - 1, "the first CTA after the scanner codes");
constexpr int kCoderWarps = kCoders / 32;
constexpr unsigned kScanPerWarp = 32 * kScanPerLane;
// Launch modes.  kPlain: e0 supplied, or (auto) read from the statistics kernel before it.
// kSpeculative (auto, first after the workspace is cleared): every CTA takes the same sample and
// guesses e0 from it (spec_guess); when the guess is confident, code with it and sum the squares
// while coding -- the CTA whose chunks complete the count checks the guess against the exact
// rule on the whole tensor's sum and sets the fallback word when it differs (or cannot be
// settled); when it is not, set the fallback word and leave.  kGated: after the gated
// statistics kernel; runs as kPlain (auto) only when the fallback word is set, else returns.
constexpr int kPlain = 0, kSpeculative = 1, kGated = 2;
static_assert(kPlain == 0, "launch_encode's default mode is kPlain");

struct EncodeParams {
  const uint16_t* in;
  uint64_t n;
  uint64_t N;
  uint8_t* out;
  Control* ctrl;
  unsigned long long* flags;
  unsigned long long* out_bytes;
  int base;  // -1: read e0 from the control block
  int* status;
  uint64_t stall_chunk;
  unsigned spin_limit;
  uint64_t full_chunks;  // n / 4096: chunks that come by one tiled copy each
  uint16_t* values;      // loopback: the decoded values (n x u16); null for compression alone
  int mode;              // kPlain, kSpeculative or kGated
};

struct __align__(128) EncodeSmem {
  uint4 xin[kStages][kInBytes / 16];
  uint4 ring[kRingBytes / 16];
  uint64_t mbar[kStages];
  unsigned ticket[kStages];
  // Escape lists in the ring, a single-producer (coding thread 0) single-consumer (retiring
  // warp) queue.  Entry i (mod kQueue): chunk, ring offset, size, bytes skipped before it.
  unsigned long long q_chunk[kQueue];
  unsigned q_off[kQueue], q_size[kQueue], q_gap[kQueue];
  volatile unsigned q_pushed;   // entries made (producer)
  volatile unsigned q_retired;  // entries written out and read back from the ring (consumer)
  volatile unsigned freed;      // ring bytes given back, gaps included (consumer)
  volatile int coders_done;     // no more entries will come
  volatile int retirer_done;    // the retiring warp has left: the ring is free
  __align__(16) unsigned scan[kCoderWarps];  // per coding warp: its escape count
  // scanner: per round parity, each warp's ready count and sum, and the status word
  unsigned long long scan_sum[2][kCoderWarps];
  unsigned scan_ready[2][kCoderWarps];
  int scan_bad[2];
  int e0;
  int skip;       // nothing to code: the raw pass wrote the stream, or the first phase failed
  int kind;       // the first phase's job: 0 none, 1 the exact e0, 2 the raw pass
  int first_ok;   // the first phase ended with its result published
  int first_last; // this CTA finished the first phase's last chunk
  unsigned role;  // 0: this CTA scans; otherwise it codes (and, in the loopback, decodes)
  // loopback decoding: the chunk, its escape section and the code-7 count
  unsigned dchunk;
  unsigned long long doff;
  unsigned dsize;
  int dok;
  unsigned descapes;
  unsigned slot_chunk[2], slot_size[2];  // a decoding CTA's two slots
  int slot_ok[2];
  unsigned lb_parity;  // a coding CTA turned decoder: the stages' mbarrier phases to wait for next
  // speculative: the coding warps' sums, and whether this CTA completed the chunk count
  double spec_sum[kCoderWarps];
  unsigned long long spec_nf[kCoderWarps], spec_values[kCoderWarps], spec_inside[kCoderWarps];
  int spec_last;
  int spec;       // this launch speculates (kSpeculative, and the sample was confident)
  // the sample's per-warp sums (scaled by 2^(126 - Es)), finite counts and escapes under the guess
  float g2[kCoderWarps], g4[kCoderWarps];
  int gk[kCoderWarps];
  unsigned gf[kCoderWarps], gesc[kCoderWarps];
  int guess;
  int confident;
  int e_end[2];
};

__device__ __forceinline__ void bar_coders() { asm volatile("bar.sync 1, %0;" ::"n"(kCoders) : "memory"); }

// The coding threads' escape counts in thread order (= position order): this thread's first
// rank (the exclusive prefix) and the chunk total.  One barrier over the coding threads [R];
// `scratch` holds one word per coding warp, read as one 16-byte word.
__device__ __forceinline__ unsigned chunk_rank(unsigned cnt, unsigned* first, unsigned* scratch) {
  static_assert(kCoderWarps == 4, "one 16-byte read of the warp totals");
  const unsigned lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned x = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned t = __shfl_up_sync(0xFFFFFFFFu, x, o);
    if (lane >= static_cast<unsigned>(o)) x += t;
  }
  if (lane == 31) scratch[warp] = x;
  bar_coders();
  const uint4 tw = *reinterpret_cast<const uint4*>(scratch);
  const unsigned before = (warp > 0 ? tw.x : 0u) + (warp > 1 ? tw.y : 0u) + (warp > 2 ? tw.z : 0u);
  *first = before + x - cnt;
  return tw.x + tw.y + tw.z + tw.w;
}

// Ask for `bytes` (a multiple of 16) at a 16-byte aligned global address to be brought into L2.
__device__ __forceinline__ void prefetch_l2(const void* p, unsigned bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Coding thread 0: start the copy of chunk c into stage s.  A full chunk is one box of the
// input's tensor map, written to shared memory with the 128-byte swizzle (16-byte unit u of
// 128-byte row r lands at unit u ^ (r % 8)), so that each coding thread's four 16-byte reads of
// its own 64 bytes meet no bank twice.  The ragged last chunk comes without a copy: every coding
// thread fetches its own values.
__device__ void issue_load(EncodeSmem& S, int s, uint64_t c, const EncodeParams& p, const CUtensorMap* map) {
  if (c < p.full_chunks) {
    mbar_arrive_expect_tx(&S.mbar[s], kInBytes);
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(smem_u32(S.xin[s])),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(0), "r"(static_cast<int>(c)), "r"(smem_u32(&S.mbar[s]))
        : "memory");
  } else {
    mbar_arrive(&S.mbar[s]);
  }
}

// The scanner (the first CTA to start, its kCoderWarps first warps): resolve chunks in order.
// Each round, warp w reads state words frontier + 256 w .. + 255; the published sizes before
// the first unpublished word (over all warps, in order) become inclusive offsets.  One barrier
// per round exchanges the warps' ready counts and sums (double-buffered by round parity, so one
// barrier suffices).
__device__ __noinline__ void scanner(EncodeSmem& S, unsigned long long* flags, uint64_t N, int* status,
                                     unsigned spin_limit) {
  const unsigned lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint64_t frontier = 0;
  unsigned long long prefix = 0;
  unsigned spins = 0, backoff = 32;
  for (unsigned round = 0; frontier < N; ++round) {
    const unsigned b = round & 1;
    const uint64_t wbase = frontier + static_cast<uint64_t>(kScanPerWarp) * warp;
    const int bad = warp == 0 && lane == 0 ? read_status(status) : 0;  // in flight with the flags
    unsigned long long f[kScanPerLane];
#pragma unroll
    for (int j = 0; j < kScanPerLane; ++j) {
      const uint64_t idx = wbase + kScanPerLane * lane + j;
      f[j] = idx < N ? ld_relaxed_u64(&flags[idx]) : 0ull;
    }
    unsigned mine = kScanPerWarp;  // first unpublished position held by this lane
#pragma unroll
    for (int j = kScanPerLane - 1; j >= 0; --j)
      if ((f[j] >> 62) == 0) mine = kScanPerLane * lane + j;
    const unsigned ready = __reduce_min_sync(0xFFFFFFFFu, mine);
    unsigned long long own = 0;
#pragma unroll
    for (int j = 0; j < kScanPerLane; ++j)
      if (kScanPerLane * lane + j < ready) own += f[j] & kFlagValueMask;
    unsigned long long run = own;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long t = __shfl_up_sync(0xFFFFFFFFu, run, o);
      if (lane >= static_cast<unsigned>(o)) run += t;
    }
    if (lane == 31) {
      S.scan_ready[b][warp] = ready;
      S.scan_sum[b][warp] = run;
    }
    if (warp == 0 && lane == 0) S.scan_bad[b] = bad;
    bar_coders();
    // Lanes below kCoderWarps hold the warps' results; warps before the first partly ready one are
    // whole, and that one contributes its ready part.
    const unsigned r8 = lane < kCoderWarps ? S.scan_ready[b][lane] : 0u;
    const unsigned long long s8 = lane < kCoderWarps ? S.scan_sum[b][lane] : 0ull;
    const unsigned whole = __ballot_sync(0xFFFFFFFFu, lane < kCoderWarps && r8 == kScanPerWarp);
    const unsigned first_partial = __ffs(~whole) - 1;  // kCoderWarps when all are whole
    const unsigned tail_ready = __shfl_sync(0xFFFFFFFFu, r8, first_partial & 31);
    const uint64_t total_ready = static_cast<uint64_t>(kScanPerWarp) * first_partial +
                                 (first_partial < static_cast<unsigned>(kCoderWarps) ? tail_ready : 0u);
    const unsigned long long use = lane <= first_partial ? s8 : 0ull;  // sums that count
    unsigned long long before = lane < warp ? use : 0ull, total = use;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      before += __shfl_xor_sync(0xFFFFFFFFu, before, o);
      total += __shfl_xor_sync(0xFFFFFFFFu, total, o);
    }
    if (total_ready == 0) {
      if (S.scan_bad[b] != 0) return;
      if (++spins > spin_limit) {
        if (warp == 0 && lane == 0) set_error(status, ZC_ERR_TIMEOUT);
        return;
      }
      __nanosleep(backoff);
      backoff = backoff < 256 ? backoff * 2 : 256;
      continue;
    }
    spins = 0;
    backoff = 32;
    if (warp <= first_partial) {
      unsigned long long acc = prefix + before + (run - own);
#pragma unroll
      for (int j = 0; j < kScanPerLane; ++j) {
        const unsigned q = kScanPerLane * lane + j;
        if (q < ready) {
          acc += f[j] & kFlagValueMask;
          st_relaxed_u64(&flags[wbase + q], kFlagInclusive | acc);
        }
      }
    }
    prefix += total;
    frontier += total_ready;
  }
}

// The retiring warp: copy escape sections out in chunk order as the scanner resolves them, fill in
// the offset table (and the header fields that belong to the first and last chunk), and give
// the ring space back.  Lists and their places are 16-byte aligned, so the whole warp copies
// each one with 16-byte loads and stores: plain stores, so the coding threads need no proxy
// fence before handing a list over.  Every value that steers the warp is made uniform over its
// lanes: each lane reads it itself and the warp takes the minimum (or any / all).
__device__ void retirer(EncodeSmem& S, const EncodeParams& p) {
  const unsigned lane = threadIdx.x & 31;
  const uint64_t E0 = escape_base(p.n);
  // A section ending past the raw form's length means the stream will be raw: it is not written
  // (except in the loopback, which decodes every section of the coded form).
  const uint64_t room = p.values ? ~0ull : raw_stream_bytes(p.n) > E0 ? raw_stream_bytes(p.n) - E0 : 0;
  unsigned long long* table = reinterpret_cast<unsigned long long*>(p.out + kHeaderBytes);
  unsigned retired = 0, freed = 0, spins = 0, backoff = 64;
  for (;;) {
    const unsigned pushed = __reduce_min_sync(0xFFFFFFFFu, S.q_pushed);
    const unsigned avail = pushed - retired;
    if (avail == 0) {
      if (__all_sync(0xFFFFFFFFu, S.coders_done != 0)) {  // q_pushed was bumped before coders_done
        __threadfence_block();
        if (__reduce_min_sync(0xFFFFFFFFu, S.q_pushed) == retired) break;
        continue;
      }
      if (__any_sync(0xFFFFFFFFu, read_status(p.status) != 0)) break;
      if (++spins > p.spin_limit) {
        if (lane == 0) set_error(p.status, ZC_ERR_TIMEOUT);
        break;
      }
      __nanosleep(backoff);
      backoff = backoff < 512 ? backoff * 2 : 512;
      continue;
    }
    __threadfence_block();  // the entries below were written before q_pushed was bumped
    const unsigned i = (retired + lane) % kQueue;
    const bool mine = lane < avail;
    const unsigned long long f = mine ? ld_relaxed_u64(&p.flags[S.q_chunk[i]]) : 0ull;
    const unsigned resolved = __ballot_sync(0xFFFFFFFFu, mine && (f >> 62) == 2);
    const unsigned run = __ffs(~resolved) ? __ffs(~resolved) - 1 : 32;  // leading resolved entries
    if (run == 0) {
      int bad = lane == 0 ? read_status(p.status) : 0;
      bad = __shfl_sync(0xFFFFFFFFu, bad, 0);
      if (bad != 0) break;
      if (++spins > p.spin_limit) {
        if (lane == 0) set_error(p.status, ZC_ERR_TIMEOUT);
        break;
      }
      __nanosleep(backoff);
      backoff = backoff < 512 ? backoff * 2 : 512;
      continue;
    }
    spins = 0;
    backoff = 64;
    for (unsigned t = 0; t < run; ++t) {  // the lists, in order, each by the whole warp
      const unsigned long long ft = __shfl_sync(0xFFFFFFFFu, f, t);
      if ((ft & kFlagValueMask) > room) break;  // this one and all later ones: the stream is raw
      const unsigned it = (retired + t) % kQueue;
      const unsigned size = S.q_size[it];
      const uint4* src = S.ring + S.q_off[it] / 16;
      uint4* dst = reinterpret_cast<uint4*>(p.out + E0 + (ft & kFlagValueMask) - size);
      for (unsigned v = lane; v < size / 16; v += 32) dst[v] = src[v];
    }
    unsigned give_back = 0;
    if (lane < run) {
      const unsigned long long c = S.q_chunk[i];
      const unsigned size = S.q_size[i];
      const unsigned long long off = E0 + (f & kFlagValueMask) - size;
      table[c] = off;
      if (c == 0) {
        unsigned long long* hdr = reinterpret_cast<unsigned long long*>(p.out);
        hdr[0] = kMagicWord | (static_cast<unsigned long long>(S.e0) << 56);
        hdr[1] = p.n;
        hdr[2] = p.N;
        if (kHeaderBytes + 8 * (p.N + 1) < records_base(p.n)) table[p.N + 1] = 0;  // zero pad
      }
      if (c == p.N - 1) {
        const unsigned long long total = off + size;
        table[p.N] = total;
        reinterpret_cast<unsigned long long*>(p.out)[3] = total;
        p.ctrl->total = total;
        if (p.out_bytes) *p.out_bytes = total;
      }
      give_back = S.q_gap[i] + size;
    }
    if (p.values) {
      // Loopback: the sections and offsets above are written; mark each chunk copied, so that a
      // decoding CTA may take it (the fence orders the warp's stores, and the coding threads'
      // fixed parts that reached this warp through the queue, before the mark).
      __syncwarp();
      if (lane < run) {
        __threadfence();
        st_relaxed_u64(&p.flags[S.q_chunk[i]], kFlagCopied | (f & kFlagValueMask));
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) give_back += __shfl_xor_sync(0xFFFFFFFFu, give_back, o);
    retired += run;
    freed += give_back;
    __syncwarp();
    if (lane == 0) {
      __threadfence_block();  // the copies have read the ring before it is handed back
      S.freed = freed;
      S.q_retired = retired;
    }
    __syncwarp();
  }
  __syncwarp();  // every lane's copies out of the ring are done
  if (lane == 0) {
    __threadfence_block();
    S.retirer_done = 1;
  }
}

// The ring as every coding thread tracks it (the same in all of them, so each can place the
// next list itself): `need` bytes (a multiple of 16, at most kMaxEscapeBytes) at `where`, after
// skipping `gap` bytes at the end.
struct Ring {
  unsigned pushed = 0;  // entries made
  unsigned made = 0;    // ring bytes handed out, gaps included
  unsigned head = 0;    // ring offset where the next list may start
};

// Wait (bounded) until the retiring warp has freed room for a section of `need` bytes after a
// `gap` (ring_fits) and a queue slot.  False after an error or a timeout.
__device__ bool ring_room(const EncodeSmem& S, const Ring& R, unsigned gap, unsigned need, const EncodeParams& p) {
  unsigned spins = 0, backoff = 64;
  while (R.pushed - S.q_retired >= kQueue || !ring_fits(R.made - S.freed, gap, need, kRingBytes)) {
    if (read_status(p.status) != 0) return false;
    if (++spins > p.spin_limit) {
      set_error(p.status, ZC_ERR_TIMEOUT);
      return false;
    }
    __nanosleep(backoff);
    backoff = backoff < 512 ? backoff * 2 : 512;
  }
  return true;
}

// An exponent plane: this thread's 32 exponent bytes at `dst` (shared window; byte v0 of the
// section), read back from the staged input (values past m are zero there, so the section's
// padding comes out zero); `room` bytes of the section lie at or past dst.  Out of line, off
// the path of chunks with a list.
__device__ __noinline__ void write_plane(const uint4* stage, unsigned sw, uint32_t dst, unsigned room) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint4 xv = stage[(sw ^ (16 * q)) / 16];
    const uint32_t lo = prmt((xv.x >> 7) & 0x00FF00FFu, (xv.y >> 7) & 0x00FF00FFu, 0x6420);
    const uint32_t hi = prmt((xv.z >> 7) & 0x00FF00FFu, (xv.w >> 7) & 0x00FF00FFu, 0x6420);
    if (8u * q < room) sts_v2(dst + 8 * q, lo, hi);
  }
}

// ------------------------------------------------------------------ the first phase
//
// In auto mode the statistics pass may leave one of two jobs, done here before any chunk is
// coded.  Their chunks are handed out by a ticket of their own, in batches to a warp; each CTA
// adds its results and the number of chunks it finished to the control block, and the CTA whose
// count completes N finishes the job and publishes it (first_ready, a release store); the others
// wait for that, bounded.  A CTA waits only on chunks that a running CTA has taken, so the phase
// needs no CTA to be resident at any particular time.
//  - Exact e0 (kind 1), when the statistics pass's estimate could not settle it: every thread sums
//    sig^2 4^d exactly in a 128-bit integer over a 24-binade window from Eb (around the typical
//    value, anchored on the estimate's e0; a term is below 2^62, so 2^66 of them fit); values
//    outside the window add sig^2 to their exponent's bin in shared memory.  The finisher rounds
//    the 576-bit total of the grid's bins and window sums once to fp64 and picks e0
//    (exact_from_bins, select_e0).
//  - Raw pass (kind 2), when the statistics pass's exponent sample predicted a raw stream (the
//    third technique: the native path when coding does not pay): every value is copied to its
//    place in the raw form and every chunk's escapes are counted under e0 exactly as the coding
//    counts them, giving its escape section's size.  The finisher compares the coded form's
//    exact length with the raw form's; when the coded one is longer it completes the raw form
//    (header, length) and marks the stream done, so nothing is coded.  Otherwise (ties included)
//    the coding writes the coded form over the copy.
constexpr int kFirstVecPerLane = kChunk / 8 / 32;  // 16 vectors of a chunk per lane
constexpr unsigned kFirstBatch = 8;                // chunks a warp takes per ticket, at most

// Escapes among the two values of w outside `keep`'s cleared halves (codes7_x2 gives exactly
// 7 << 7 for an escape, and 7 << 7 + 0x80 reaches bit 10).
__device__ __forceinline__ unsigned escapes_x2(uint32_t w, uint32_t kadd, uint32_t keep = 0xFFFFFFFFu) {
  return __popc(((codes7_x2(w, kadd) & keep) + 0x00800080u) & 0x04000400u);
}

// Raw pass, one warp: chunk c's values copied behind the 32-byte header (the last vector of the
// stream completed with zeros); returns the chunk's escape-section bytes in every lane.
__device__ unsigned raw_chunk(const uint16_t* x, uint64_t n, uint64_t c, uint32_t kadd, uint8_t* out) {
  const unsigned lane = threadIdx.x & 31;
  const uint4* src = reinterpret_cast<const uint4*>(x);
  uint4* dst = reinterpret_cast<uint4*>(out + kHeaderBytes);
  const uint64_t nv = n / 8;
  unsigned esc = 0, m = kChunk;
  if (c < n / kChunk) {
#pragma unroll 1
    for (int h = 0; h < 2; ++h) {  // two halves of 8 vectors per lane
      const uint64_t b = c * (kChunk / 8) + 32 * (kFirstVecPerLane / 2) * h + lane;
      uint4 v[kFirstVecPerLane / 2];
#pragma unroll
      for (int j = 0; j < kFirstVecPerLane / 2; ++j) v[j] = __ldcs(src + b + 32 * j);
#pragma unroll
      for (int j = 0; j < kFirstVecPerLane / 2; ++j) {
        __stcs(dst + b + 32 * j, v[j]);
        esc += escapes_x2(v[j].x, kadd) + escapes_x2(v[j].y, kadd) + escapes_x2(v[j].z, kadd) +
               escapes_x2(v[j].w, kadd);
      }
    }
  } else {  // the ragged last chunk: its m values
    m = static_cast<unsigned>(n - c * kChunk);
    for (unsigned i = lane; i < (m + 7) / 8; i += 32) {
      const uint64_t g = c * (kChunk / 8) + i;
      uint32_t w[4];
      if (g < nv) {
        const uint4 t = __ldcs(src + g);
        w[0] = t.x, w[1] = t.y, w[2] = t.z, w[3] = t.w;
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint64_t v = 8 * g + 2 * q;
          w[q] = (v < n ? static_cast<uint32_t>(x[v]) : 0u) | (v + 1 < n ? static_cast<uint32_t>(x[v + 1]) << 16 : 0u);
        }
      }
      __stcs(dst + g, make_uint4(w[0], w[1], w[2], w[3]));
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const unsigned v = 8 * i + 2 * q;
        esc += escapes_x2(w[q], kadd, (v < m ? 0x0000FFFFu : 0u) | (v + 1 < m ? 0xFFFF0000u : 0u));
      }
    }
  }
  const unsigned k = __reduce_add_sync(0xFFFFFFFFu, esc);
  return 3 * k <= m ? static_cast<unsigned>(pad16(3 * k)) : static_cast<unsigned>(pad16(m));
}

// Exact sums, one warp: chunk c's values (zeros past n add nothing), two at a time
// (ExactWindow); the chunk's 96-bit window sum is folded into the thread's 128-bit (lo, hi) at
// its end.
__device__ void exact_chunk(const uint16_t* x, uint64_t n, uint64_t c, int Eb, unsigned long long& lo,
                            unsigned long long& hi, unsigned long long* bins) {
  const unsigned lane = threadIdx.x & 31;
  ExactWindow ew(Eb);
  auto add_word = [&](uint32_t w) { ew.add_word(w, bins); };
  const uint4* src = reinterpret_cast<const uint4*>(x);
  const uint64_t nv = n / 8, first = c * (kChunk / 8);
  const uint64_t end = first + kChunk / 8 < nv ? first + kChunk / 8 : nv;  // whole vectors of the chunk
  constexpr int kUnroll = 4;  // 16-byte loads in flight per lane (8 was slower)
  for (uint64_t g = first + lane; g < end; g += 32 * kUnroll) {
    uint4 v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) v[u] = g + 32 * u < end ? __ldcs(src + g + 32 * u) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      add_word(v[u].x);
      add_word(v[u].y);
      add_word(v[u].z);
      add_word(v[u].w);
    }
  }
  if (c == (n - 1) / kChunk && lane < n % 8) add_word(x[8 * nv + lane]);  // the last n % 8 values
  // 128 terms per lane at most, each below 2^62: the chunk's sum fits in 96 bits
  const unsigned long long s = (static_cast<unsigned long long>(ew.a1) << 32) | ew.a0;
  lo += s;
  hi += ew.a2 + (lo < s);
}

// Bounded wait (one thread) for the first phase's result.  False after an error or a timeout.
__device__ bool wait_first_ready(Control* ctrl, int* status, unsigned spin_limit) {
  unsigned spins = 0, backoff = 64;
  while (ld_acquire_u32(&ctrl->first_ready) == 0) {
    if (read_status(status) != 0) return false;
    if (++spins > spin_limit) {
      set_error(status, ZC_ERR_TIMEOUT);
      return false;
    }
    __nanosleep(backoff);
    backoff = backoff < 512 ? backoff * 2 : 512;
  }
  return true;
}

// The first phase, by the 128 coding threads of a CTA.  Returns (in every thread) whether the
// result is published; e0 and the stream form are then final in the control block.
__device__ __noinline__ bool first_phase(EncodeSmem& S, const uint16_t* x, uint64_t n, uint64_t N, uint8_t* out,
                                         unsigned long long* out_bytes, Control* ctrl, unsigned long long* gbins,
                                         int* status, unsigned spin_limit, int kind) {
  const unsigned tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  unsigned long long* bins = reinterpret_cast<unsigned long long*>(S.ring);  // exact: this CTA's bins
  unsigned long long* pieces = S.scan_sum[1];                               // exact: its window sums
  if (kind == 1) {
    for (unsigned i = tid; i < 256; i += kCoders) bins[i] = 0;
    if (tid < 4) pieces[tid] = 0;
  }
  bar_coders();
  const int e0 = __ldcg(&ctrl->e0);
  const uint32_t kadd = ((256u - static_cast<unsigned>(e0)) << 7) * 0x00010001u;
  int Eb = e0 - 12;  // e0 + 5 is about the typical exponent of a Gaussian tensor
  Eb = Eb < 1 ? 1 : (Eb > 254 - kExactWindow ? 254 - kExactWindow : Eb);
  unsigned long long lo = 0, hi = 0, bytes = 0;
  unsigned mine = 0;  // chunks this warp finished
  // Batches of chunks per ticket (fewer atomics on the one counter): about a quarter of what is
  // left per warp, so the batches shrink to one chunk as the tickets run out and the last ones
  // end together.  Each chunk is brought into L2 by one bulk prefetch two chunks ahead.
  const uint64_t warps = static_cast<uint64_t>(gridDim.x) * kCoderWarps;
  unsigned seen = 0;  // the ticket counter as this warp last saw it
  for (;;) {
    const uint64_t left = N > seen ? N - seen : 0;
    const unsigned batch = left > 4 * kFirstBatch * warps ? kFirstBatch
                                                          : static_cast<unsigned>(left / (4 * warps)) + 1;
    unsigned c0 = 0;
    if (lane == 0) c0 = atomicAdd(&ctrl->first_ticket, batch);
    c0 = __shfl_sync(0xFFFFFFFFu, c0, 0);
    if (c0 >= N) break;
    seen = c0 + batch;
    const unsigned cend = c0 + batch < N ? c0 + batch : static_cast<unsigned>(N);
    const uint64_t full = n / kChunk;  // whole chunks: 8 KiB each, 16-byte aligned
    auto prefetch = [&](uint64_t c) { prefetch_l2(x + c * kChunk, 2 * kChunk); };
    if (lane < 2 && c0 + lane < cend && c0 + lane < full) prefetch(c0 + lane);
    for (unsigned c = c0; c < cend; ++c) {
      if (lane == 0 && c + 2 < cend && c + 2 < full) prefetch(c + 2);
      if (kind == 2)
        bytes += raw_chunk(x, n, c, kadd, out);
      else
        exact_chunk(x, n, c, Eb, lo, hi, bins);
      ++mine;
    }
  }
  if (kind == 1) {  // the window sums in 32-bit pieces, over the warp, then the CTA
    unsigned long long pc[4] = {lo & 0xFFFFFFFFull, lo >> 32, hi & 0xFFFFFFFFull, hi >> 32};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) pc[k] += __shfl_xor_sync(0xFFFFFFFFu, pc[k], o);
      if (lane == 0 && pc[k]) atomicAdd(pieces + k, pc[k]);
    }
  }
  if (lane == 0) {
    S.scan_sum[0][warp] = bytes;
    S.scan_ready[0][warp] = mine;
  }
  bar_coders();
  // The CTA's results into the grid's, each thread's made visible (fence) before the CTA reports
  // its chunks; the report that completes N makes this CTA the finisher.
  if (kind == 1) {
    for (unsigned i = tid; i < 256; i += kCoders)
      if (bins[i]) atomicAdd(gbins + i, bins[i]);
    if (tid < 4 && pieces[tid]) atomicAdd(&ctrl->exact_pieces[tid], pieces[tid]);
  } else if (tid == 0) {
    unsigned long long sum = 0;
    for (int w = 0; w < kCoderWarps; ++w) sum += S.scan_sum[0][w];
    if (sum) atomicAdd(&ctrl->raw_escape_bytes, sum);
  }
  __threadfence();
  bar_coders();
  if (tid == 0) {
    unsigned count = 0;
    for (int w = 0; w < kCoderWarps; ++w) count += S.scan_ready[0][w];
    S.first_last = count != 0 && atomicAdd(&ctrl->first_done, count) == N - count;
    if (S.first_last) __threadfence();  // acquire: every CTA's results are visible from here on
  }
  bar_coders();
  if (S.first_last) {
    if (kind == 1) {
      for (unsigned i = tid; i < 256; i += kCoders) bins[i] = __ldcg(gbins + i);
      if (tid < 4) pieces[tid] = __ldcg(&ctrl->exact_pieces[tid]);
      bar_coders();
      if (tid == 0) ctrl->e0 = select_e0(exact_from_bins(bins, pieces, Eb), __ldcg(&ctrl->n_finite));
    } else if (tid == 0) {
      const unsigned long long coded = escape_base(n) + __ldcg(&ctrl->raw_escape_bytes), raw = raw_stream_bytes(n);
      if (coded > raw) {
        unsigned long long* hdr = reinterpret_cast<unsigned long long*>(out);
        hdr[0] = kRawMagicWord | (static_cast<unsigned long long>(e0) << 56);
        hdr[1] = n;
        hdr[2] = 0;
        hdr[3] = raw;
        ctrl->total = raw;
        if (out_bytes) *out_bytes = raw;
        ctrl->raw_done = 1;
      }
    }
    if (tid == 0) {
      __threadfence();
      st_release_u32(&ctrl->first_ready, 1u);
      S.first_ok = 1;
    }
  } else if (tid == 0) {
    S.first_ok = wait_first_ready(ctrl, status, spin_limit) ? 1 : 0;
  }
  bar_coders();
  return S.first_ok != 0;
}

__device__ __forceinline__ bool bar_coders_or(bool v) {
  unsigned r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\t"
      "bar.red.or.pred p, 1, %2, q;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"(static_cast<unsigned>(v)), "n"(kCoders)
      : "memory");
  return r != 0;
}

// The escape section of a chunk marked copied (state word f, read before an acquire fence): its
// offset from the offset table (written by the same retiring lane before its fence and the mark,
// so visible after the acquire; the state word of the chunk before it comes from another lane of
// the scanner and may not be), its end from f.  Every size is checked before anything is read by
// it: a section that does not fit its place sets ZC_ERR_CORRUPT and returns false.
__device__ bool copied_section(const uint8_t* stream, int* status, uint64_t E0, unsigned d, unsigned long long f,
                               unsigned long long* off, unsigned* size) {
  const unsigned long long end = E0 + (f & kFlagValueMask);
  const unsigned long long o = __ldcg(reinterpret_cast<const unsigned long long*>(stream + kHeaderBytes) + d);
  if (o < E0 || o > end || end - o > kMaxEscapeBytes || ((end - o) & 15u) != 0) {
    set_error(status, ZC_ERR_CORRUPT);
    return false;
  }
  *off = o;
  *size = static_cast<unsigned>(end - o);
  return true;
}

// Loopback decoding: chunks are decoded in ticket order as their escape sections reach the
// stream (the split-send pipeline: a chunk is transmissible, and here decoded, as soon as its own
// bytes are in place, while later chunks are still being coded).  Each chunk waits (bounded,
// thread 0) for its copied mark, then its fixed part and escape section are read back from the
// stream and decoded with the decode kernel's own code.
struct LoopbackArgs {  // what the loopback decoding needs, passed in registers
  const uint8_t* stream;
  uint16_t* values;
  unsigned long long* flags;
  Control* ctrl;
  int* status;
  uint64_t n, N;
  unsigned spin_limit;
};

// Thread 0: take the next chunk to decode and wait (bounded) for its copied mark.  Returns false
// when no chunk is left or after an error or a timeout; otherwise *off and *size give its escape
// section, and its bytes are visible to this thread's later reads (acquire).
__device__ bool claim_decode(const LoopbackArgs& p, uint64_t E0, unsigned* d, unsigned long long* off,
                             unsigned* size) {
  *d = atomicAdd(&p.ctrl->decode_ticket, 1u);
  if (*d >= p.N) return false;
  unsigned spins = 0, backoff = 64;
  unsigned long long f;
  while (((f = ld_relaxed_u64(&p.flags[*d])) >> 62) != 3) {
    if (read_status(p.status) != 0) return false;
    if (++spins > p.spin_limit) {
      set_error(p.status, ZC_ERR_TIMEOUT);
      return false;
    }
    __nanosleep(backoff);
    backoff = backoff < 512 ? backoff * 2 : 512;
  }
  __threadfence();  // acquire: the chunk's bytes and its offset are visible from here on
  return copied_section(p.stream, p.status, E0, *d, f, off, size);
}

// Loopback, the 128 coding threads of a CTA that decodes: two slots, each a chunk's fixed part
// (in an input stage) and escape section (in the ring), filled by bulk async copies; the next
// chunk's copies are in flight while a chunk is decoded.  A CTA that only decodes starts here
// (fresh mbarriers); a coding CTA comes here once it has no chunk left to code and its retiring
// warp has left (the ring is free), reusing the stages' mbarriers from the phases in
// S.lb_parity (`reuse`).
__device__ __noinline__ void loopback_decode_slots(EncodeSmem& S, const uint8_t* stream, uint16_t* values,
                                                   unsigned long long* flags, Control* ctrl, int* status, uint64_t n,
                                                   uint64_t N, unsigned spin_limit, bool reuse) {
  const LoopbackArgs p{stream, values, flags, ctrl, status, n, N, spin_limit};
  const unsigned tid = threadIdx.x;
  const uint64_t E0 = escape_base(p.n), R0 = records_base(p.n);
  // slot j: fixed part in input stage j, escape section in the ring at 4096 j
  auto fixed_of = [&](int j) { return S.xin[0] + j * (kInBytes / 16); };
  auto esc_of = [&](int j) { return S.ring + j * (kMaxEscapeBytes / 16); };
  // thread 0: claim a chunk and start its copies into slot j
  auto fill = [&](int j) {
    unsigned d = 0, size = 0;
    unsigned long long off = 0;
    const bool ok = claim_decode(p, E0, &d, &off, &size);
    S.slot_chunk[j] = d;
    S.slot_size[j] = size;
    S.slot_ok[j] = ok;
    if (ok) {
      const unsigned fb = static_cast<unsigned>(fixed_bytes(chunk_values(p.n, d)));
      asm volatile("fence.proxy.async.global;" ::: "memory");  // the acquired bytes, for the copy engine
      mbar_arrive_expect_tx(&S.mbar[j], fb + size);
      bulk_load(fixed_of(j), p.stream + R0 + static_cast<uint64_t>(d) * kFullFixedBytes, fb, &S.mbar[j]);
      if (size) bulk_load(esc_of(j), p.stream + off, size, &S.mbar[j]);
    }
  };
  if (tid == 0) {
    if (!reuse) {
      for (int j = 0; j < 2; ++j) mbar_init(&S.mbar[j], 1);
      fence_mbar_init();
    }
    fill(0);
    fill(1);
  }
  bar_coders();
  unsigned parity = reuse ? S.lb_parity : 0u;
  for (int j = 0;; j ^= 1) {
    if (!S.slot_ok[j]) break;
    // every thread polls; all act on one shared answer
    const bool arrived = mbar_wait(&S.mbar[j], (parity >> j) & 1u, kWaitLimit);
    parity ^= 1u << j;
    if (bar_coders_or(!arrived)) {
      if (tid == 0) {  // never leave a copy in flight (bounded again)
        set_error(p.status, ZC_ERR_TIMEOUT);
        mbar_wait(&S.mbar[j], ((parity >> j) & 1u) ^ 1u, kWaitLimit);
        if (S.slot_ok[j ^ 1]) mbar_wait(&S.mbar[j ^ 1], (parity >> (j ^ 1)) & 1u, kWaitLimit);
      }
      return;
    }
    const unsigned d = S.slot_chunk[j];
    if (tid == 0) S.descapes = 0;
    bar_coders();
    decode_chunk(fixed_of(j), esc_of(j), &S.descapes, p.values + static_cast<uint64_t>(d) * kChunk,
                 chunk_values(p.n, d), S.e0, S.slot_size[j], p.status, tid, [] { bar_coders(); });
    bar_coders();  // slot j is read: refill it
    if (tid == 0) fill(j);
    bar_coders();
  }
  // the other slot may still hold a claimed chunk whose copies are in flight: decode it too
  const int k = S.slot_ok[0] ? 0 : (S.slot_ok[1] ? 1 : -1);
  if (k >= 0) {
    const bool arrived = mbar_wait(&S.mbar[k], (parity >> k) & 1u, kWaitLimit);
    if (bar_coders_or(!arrived)) {
      if (tid == 0) {
        set_error(p.status, ZC_ERR_TIMEOUT);
        mbar_wait(&S.mbar[k], (parity >> k) & 1u, kWaitLimit);  // never leave a copy in flight
      }
      return;
    }
    if (tid == 0) S.descapes = 0;
    bar_coders();
    const unsigned d = S.slot_chunk[k];
    decode_chunk(fixed_of(k), esc_of(k), &S.descapes, p.values + static_cast<uint64_t>(d) * kChunk,
                 chunk_values(p.n, d), S.e0, S.slot_size[k], p.status, tid, [] { bar_coders(); });
  }
}

// Speculative mode: one coding thread's share of a chunk's sum of squares, its 32 values (xv) as
// one block.  With e0 in [kFastE0Min, kFastE0Max] (`fast`), the values inside the window have
// magnitudes in [2^-40, 2^61), so their squares are normal fp32 numbers, and the block is summed
// plainly: bf16 -> fp32 by a shift or a mask, squares by packed fp32x2 FMAs into four partial
// sums (at most 11 roundings, relative error below 2^-19 while nothing underflows).  An escape can
// overflow (the sum is then not finite, as it is for Inf and NaN inputs): such a lane's block goes
// through block_sum, the careful sum.  An escape can also underflow, losing at most 2^-150 per
// operation; against a sum of squares of which half the values lie inside the window (each
// square at least 2^-80), that is below 2^-66 of it -- so the CTA checks that half of its values
// were inside the window (spec_verdict), and otherwise the guess is not trusted.  Outside that
// range of e0 every block goes through block_sum.
constexpr int kFastE0Min = 87, kFastE0Max = 180;

__device__ __forceinline__ unsigned long long fma_f32x2(unsigned long long a, unsigned long long b,
                                                        unsigned long long c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

__device__ __forceinline__ void spec_square_sum(const uint4 (&xv)[4], bool fast, double* acc, unsigned* nonfinite) {
  const uint32_t w[16] = {xv[0].x, xv[0].y, xv[0].z, xv[0].w, xv[1].x, xv[1].y, xv[1].z, xv[1].w,
                          xv[2].x, xv[2].y, xv[2].z, xv[2].w, xv[3].x, xv[3].y, xv[3].z, xv[3].w};
  bool redo = !fast;
  if (fast) {
    unsigned long long a = 0, b = 0;  // two fp32x2 accumulators: four partial sums
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const unsigned long long x =
          static_cast<unsigned long long>(w[i] << 16) | (static_cast<unsigned long long>(w[i] & 0xFFFF0000u) << 32);
      if (i & 1) b = fma_f32x2(x, x, b);
      else a = fma_f32x2(x, x, a);
    }
    const float s = (__uint_as_float(static_cast<uint32_t>(a)) + __uint_as_float(static_cast<uint32_t>(a >> 32))) +
                    (__uint_as_float(static_cast<uint32_t>(b)) + __uint_as_float(static_cast<uint32_t>(b >> 32)));
    redo = !isfinite(s);
    if (!redo) *acc += static_cast<double>(s);
  }
  if (__any_sync(0xFFFFFFFFu, redo)) {  // block_sum's vote needs every lane: the others add zeros
    uint32_t z[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) z[i] = redo ? w[i] : 0u;
    block_sum(z, acc, nonfinite);
  }
}

// Speculative mode, the coding threads of every CTA before anything else: the guess of e0 and
// whether to trust it, from a fixed sample -- 512 chunks spread evenly over the tensor, chunk c
// giving its vector (37 c + 11) mod 512 (8 values), four vectors per thread -- which every CTA
// reads and reduces in the same order, so all reach the same guess and the same verdict without
// a word between them (after the first CTA the sample comes from the L2).  Squares and fourth
// powers in fp32, scaled by a power of two from the warp's largest magnitude; the rule's e0 at
// the sample's mean square (in fp32, the binary exponent taken out first) and at that times
// 1 -+ (4 r + 1/32), r the mean square's relative standard error estimated from the fourth
// powers.  Confident when the three agree, the sample has a finite nonzero value, and the stream
// the sample predicts under the guess (the fixed parts plus min(3p, 1) bytes per value, p its
// share of escapes) is shorter than 0.95 of the raw form.  A tensor near a switching point, one
// whose sum of squares a few large values dominate, and one that may come out raw go the safe
// way.  Leaves S.guess and S.confident.
#ifndef ZC_GUESS_VECTORS
#define ZC_GUESS_VECTORS 4
#endif
constexpr int kGuessVectors = ZC_GUESS_VECTORS;  // sampled vectors per coding thread: 512 chunks, 4096 values

__device__ __noinline__ void spec_guess(EncodeSmem& S, const EncodeParams& p) {
  const unsigned tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint4* in = reinterpret_cast<const uint4*>(p.in);
  const uint64_t full = p.full_chunks;
  uint32_t w[4 * kGuessVectors];
#pragma unroll
  for (int h = 0; h < kGuessVectors; ++h) {  // all loads in flight at once
    const uint64_t c = (static_cast<uint64_t>(tid + kCoders * h) * full) / (kCoders * kGuessVectors);
    const uint4 v = __ldg(in + c * (kChunk / 8) + ((37 * c + 11) & (kChunk / 8 - 1)));
    w[4 * h] = v.x;
    w[4 * h + 1] = v.y;
    w[4 * h + 2] = v.z;
    w[4 * h + 3] = v.w;
  }
  constexpr int kVals = 8 * kGuessVectors;  // this thread's sampled values
  guess_e0<kCoders>(w, kVals, S.g2, S.g4, S.gk, S.gf, &S.guess, &S.confident, [] { bar_coders(); });
  // the sample's escapes under the guess: the predicted stream must be clearly shorter than raw
  const unsigned g = static_cast<unsigned>(S.guess);
  unsigned esc = 0;
#pragma unroll
  for (int i = 0; i < kVals; ++i) esc += (((w[i >> 1] >> (16 * (i & 1) + 7)) & 0xFFu) - g) >= 7u;
  esc = __reduce_add_sync(0xFFFFFFFFu, esc);
  if (lane == 0) S.gesc[warp] = esc;
  bar_coders();
  if (tid == 0 && S.confident) {
    unsigned e = 0;
    for (int i = 0; i < kCoderWarps; ++i) e += S.gesc[i];
    const float per_value = fminf(3.0f * static_cast<float>(e) / static_cast<float>(kVals * kCoders), 1.0f);
    const double coded = static_cast<double>(escape_base(p.n)) + static_cast<double>(per_value) * static_cast<double>(p.n);
    S.confident = coded < 0.95 * static_cast<double>(raw_stream_bytes(p.n));
  }
  bar_coders();
}

// Speculative mode, the coding threads of a CTA after its last chunk: the CTA's sums are added to
// the control block's, and its chunks to the count.  The CTA whose chunks complete the count (an
// acquire-release add tells it; every other coding CTA added its sums before its own count)
// applies the rule to the total exactly as the statistics kernel does (decide_e0_pair: one end
// per thread), and sets the fallback word unless the rule settles the e0 the chunks were coded
// with.
// The order of the additions varies from run to run; the rule's bound holds for every order, so
// the e0 it settles does not.  A CTA that took no chunk adds nothing.
__device__ __noinline__ void spec_verdict(EncodeSmem& S, const EncodeParams& p, int e0, double acc,
                                          unsigned nonfinite, unsigned chunks, bool fast,
                                          unsigned long long values, unsigned long long inside) {
  const unsigned tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  unsigned long long nf = nonfinite;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
    nf += __shfl_xor_sync(0xFFFFFFFFu, nf, o);
    values += __shfl_xor_sync(0xFFFFFFFFu, values, o);
    inside += __shfl_xor_sync(0xFFFFFFFFu, inside, o);
  }
  if (lane == 0) {
    S.spec_sum[warp] = acc;
    S.spec_nf[warp] = nf;
    S.spec_values[warp] = values;
    S.spec_inside[warp] = inside;
  }
  bar_coders();
  if (tid == 0) {
    S.spec_last = 0;
    if (chunks != 0) {
      double s = 0.0;
      unsigned long long c = 0, v = 0, in = 0;
      for (int i = 0; i < kCoderWarps; ++i) {
        s += S.spec_sum[i];
        c += S.spec_nf[i];
        v += S.spec_values[i];
        in += S.spec_inside[i];
      }
      // The plain fp32 squares are within the bound only for a CTA with at least half of its
      // values inside the window (spec_square_sum); otherwise the guess is not trusted.
      if (fast && 2 * in < v) p.ctrl->spec_untrusted = 1u;
      atomicAdd(&p.ctrl->spec_sum, s);
      atomicAdd(&p.ctrl->spec_nonfinite, c);
      unsigned old;
      asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;"
                   : "=r"(old)
                   : "l"(&p.ctrl->spec_chunks), "r"(chunks)
                   : "memory");
      S.spec_last = old + chunks == p.N;
    }
  }
  bar_coders();
  if (!S.spec_last) return;
  if (tid < 2) {  // every CTA's sums were added before its chunks were counted
    const double S_all = __ldcg(&p.ctrl->spec_sum);
    const unsigned long long n_f = p.n - __ldcg(&p.ctrl->spec_nonfinite);
    int e = 0;
    const bool settled = decide_e0_pair(S_all, n_f, &e);
    if (tid == 0) {
      const bool held = settled && e == e0 && __ldcg(&p.ctrl->spec_untrusted) == 0;
      p.ctrl->e0 = e0;
      p.ctrl->n_finite = n_f;
      if (!held) p.ctrl->fallback = 1u;
    }
  }
}

__global__ void __launch_bounds__(kThreads, kCtasPerSm)
    encode_kernel(const EncodeParams p, const __grid_constant__ CUtensorMap in_map) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // The stages start on a 1024-byte boundary of the shared window (the period of the swizzle).
  EncodeSmem& S = *reinterpret_cast<EncodeSmem*>(smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u));
  // The step that follows (the raw-form check) may be scheduled now: it waits for this kernel's
  // completion before it reads anything.
  asm volatile("griddepcontrol.launch_dependents;");
  const unsigned tid = threadIdx.x, warp = tid >> 5;
  if (p.mode == kGated) {
    // After the speculative path: run only when the speculation fell back.  This kernel starts
    // only after every CTA of the gated statistics kernel before it has passed that kernel's
    // wait for the speculative encode kernel (and cleared its share of the workspace), or has
    // returned after it: the fallback word is final and visible by then.  When it is set, the
    // tickets and first copies below go ahead while the statistics pass finishes, and e0 is read
    // after griddepcontrol.wait, as after the statistics kernel alone.
    if (tid == 0) S.skip = ld_acquire_u32(&p.ctrl->fallback) == 0;
    __syncthreads();
    if (S.skip) return;
  }
  if (tid == 0) {
    // The first CTA to start is the scanner.  Every other CTA waits, bounded, only on work the
    // scanner or a CTA that is already running will do (chunks are handed out at run time), so
    // the call finishes whether or not all CTAs are resident at once.
    S.role = atomicAdd(&p.ctrl->role_ticket, 1u);
    S.q_pushed = 0;
    S.q_retired = 0;
    S.freed = 0;
    S.coders_done = 0;
    S.retirer_done = 0;
    S.skip = 0;
    S.spec = 0;
  }
  __syncthreads();
  if (S.role == 0) {
    if (warp < kCoderWarps) {
      if (p.mode == kSpeculative) {  // the same guess as the coding CTAs: nothing to scan without it
        spec_guess(S, p);
        if (!S.confident) return;
      } else if (p.base < 0) {  // auto mode: wait for the first phase, if there is one (it may leave the raw form)
        if (tid == 0) {
          asm volatile("griddepcontrol.wait;" ::: "memory");
          bool ok = true;
          if (__ldcg(&p.ctrl->exact_path) != 0 || __ldcg(&p.ctrl->raw_predicted) != 0)
            ok = wait_first_ready(p.ctrl, p.status, p.spin_limit);
          S.skip = !ok || __ldcg(&p.ctrl->raw_done) != 0;
        }
        bar_coders();
        if (S.skip) return;
      }
      scanner(S, p.flags, p.N, p.status, p.spin_limit);
    }
    return;
  }
  // Loopback: kLoopbackDecoders CTAs in every kLoopbackCycle decode from the start; the others
  // code, then decode too.
  const bool decode_only = p.values != nullptr && S.role % kLoopbackCycle >= kLoopbackCycle - kLoopbackDecoders;
  if (warp == kCoders / 32) {  // the retiring warp
    if (!decode_only) retirer(S, p);
    return;
  }
  if (decode_only) {  // (the loopback never takes the raw pass; the exact e0 it may need)
    if (p.mode == kSpeculative) {  // the coding CTAs' guess; no decoding without it
      spec_guess(S, p);
      if (!S.confident) return;
      if (tid == 0) S.e0 = S.guess;
    } else {
      if (tid == 0) {
        if (p.base < 0) asm volatile("griddepcontrol.wait;" ::: "memory");
        S.kind = p.base < 0 && __ldcg(&p.ctrl->exact_path) != 0 ? 1 : 0;
      }
      bar_coders();
      if (S.kind &&
          !first_phase(S, p.in, p.n, p.N, p.out, p.out_bytes, p.ctrl,
                       reinterpret_cast<unsigned long long*>(reinterpret_cast<uint8_t*>(p.ctrl) + kWsExactBinsOffset),
                       p.status, p.spin_limit, S.kind))
        return;
      if (tid == 0) S.e0 = p.base >= 0 ? p.base : __ldcg(&p.ctrl->e0);
    }
    bar_coders();
    loopback_decode_slots(S, p.out, p.values, p.flags, p.ctrl, p.status, p.n, p.N, p.spin_limit, false);
    return;
  }

  Ring R;                                // every coding thread's copy
  bool failed = false;                   // this thread gave up a bounded wait
  unsigned pending = 0, parity = 0;      // coding thread 0: loads in flight per stage, next parity
  unsigned next_ticket = 0;              // coding thread 0: the ticket for the next free stage
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&S.mbar[s], 1);
    fence_mbar_init();
    for (int s = 0; s < kStages; ++s) {
      const unsigned c = atomicAdd(&p.ctrl->encode_ticket, 1u);
      S.ticket[s] = c;
      if (c < p.N) {
        issue_load(S, s, c, p, &in_map);
        pending |= 1u << s;
      }
    }
    next_ticket = atomicAdd(&p.ctrl->encode_ticket, 1u);
    // e0 last.  In auto mode this kernel may start while the statistics kernel is finishing
    // (a programmatic dependent launch): the tickets and input copies above do not depend on
    // it, e0 does, so wait for that kernel's completion and writes first.
    if (p.base < 0 && p.mode != kSpeculative) asm volatile("griddepcontrol.wait;" ::: "memory");
    S.kind = p.base >= 0 || p.mode == kSpeculative ? 0
             : __ldcg(&p.ctrl->exact_path) != 0    ? 1
             : __ldcg(&p.ctrl->raw_predicted) != 0 ? 2
                                                   : 0;
  }
  bar_coders();
  if (p.mode == kSpeculative) spec_guess(S, p);  // (meanwhile the first chunks arrive)
  const bool first_ok =
      S.kind == 0 ||
      first_phase(S, p.in, p.n, p.N, p.out, p.out_bytes, p.ctrl,
                  reinterpret_cast<unsigned long long*>(reinterpret_cast<uint8_t*>(p.ctrl) + kWsExactBinsOffset),
                  p.status, p.spin_limit, S.kind);
  if (tid == 0) {
    if (p.mode == kSpeculative) {  // the sample's e0, if it is trusted; else the kernels after this one
      S.spec = S.confident;
      S.e0 = S.guess;
      S.skip = !S.confident;
      if (!S.confident) p.ctrl->fallback = 1u;
    } else {
      S.e0 = p.base >= 0 ? p.base : __ldcg(&p.ctrl->e0);
      S.skip = !first_ok || (p.base < 0 && __ldcg(&p.ctrl->raw_done) != 0);
    }
  }
  bar_coders();
  const int e0 = S.e0;
  const bool skip = S.skip != 0;  // nothing to code (raw form written, or a failed wait): drain the copies and leave
  const bool speculative = S.spec != 0;
  const bool spec_fast = e0 >= kFastE0Min && e0 <= kFastE0Max;  // the plain fp32 squares (spec_square_sum)
  double spec_acc = 0.0;          // speculative: this thread's sum of squares (fp32 blocks of 32 values)
  unsigned spec_nonfinite = 0;    // ... and its Inf and NaN
  unsigned spec_chunks = 0;       // ... and the chunks this CTA coded
  unsigned long long spec_values = 0, spec_inside = 0;  // ... its values, and those inside the window
  const uint32_t kadd = ((256u - static_cast<unsigned>(e0)) << 7) * 0x00010001u;
  const uint64_t R0 = records_base(p.n);
  // This thread's 64 bytes in a stage: logical 16-byte unit q (values v0 + 8q ..) of row tid / 2
  // sits at byte offset sw ^ 16q.
  const unsigned sw = 128 * (tid >> 1) + 16 * ((4 * (tid & 1)) ^ ((tid >> 1) & 7));

  for (unsigned it = 0; !skip; ++it) {
    const int s = it % kStages;
    const unsigned c = S.ticket[s];  // set at least one barrier ago
    if (c >= p.N) break;
    if (!mbar_wait(&S.mbar[s], (it / kStages) & 1, kWaitLimit)) {
      set_error(p.status, ZC_ERR_TIMEOUT);
      failed = true;  // the CTA stops at [C]
    }
    if (tid == 0) {
      pending &= ~(1u << s);
      parity ^= 1u << s;
      // The next ticket's chunk, whose tiled copy starts when this chunk is done, is brought into
      // L2 now: a third chunk in flight per CTA without a third stage or another held ticket
      // (taking a ticket earlier to prefetch two ahead measured slower).
      if (ZC_ENCODE_PREFETCH && next_ticket < p.full_chunks)
        prefetch_l2(p.in + static_cast<uint64_t>(next_ticket) * kChunk, 2 * kChunk);
    }

    // ---- code the chunk: the fixed part goes straight to its place in the stream
    const unsigned m = chunk_values(p.n, c);
    const bool full = m == kChunk;
    const unsigned cbytes = full ? kFullCodeBytes : static_cast<unsigned>(code_section_bytes(m));
    const unsigned smbytes = full ? kChunk : static_cast<unsigned>(pad16(m));
    uint8_t* fixed = p.out + R0 + c * static_cast<uint64_t>(kFullFixedBytes);

    // Thread t codes values 32t .. 32t+31, four groups of 8: its codes are the 12 bytes at 12t
    // of the code section, its sign|mantissa bytes the 32 at 32t of the plane, and its escapes
    // take consecutive ranks.
    const unsigned v0 = 32 * tid;
    if (!full) {  // the ragged last chunk came without a copy: fetch this thread's values
      const uint16_t* src = p.in + static_cast<uint64_t>(c) * kChunk;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t w4[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const unsigned v = v0 + 8 * q + 2 * i;
          w4[i] = (v < m ? static_cast<uint32_t>(src[v]) : 0u) |
                  (v + 1 < m ? static_cast<uint32_t>(src[v + 1]) << 16 : 0u);
        }
        S.xin[s][(sw ^ (16 * q)) / 16] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
      }
    }
    uint4 xv[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) xv[q] = S.xin[s][(sw ^ (16 * q)) / 16];
    if (speculative) spec_square_sum(xv, spec_fast, &spec_acc, &spec_nonfinite);
    Coded32 kd;
    code32(xv, kadd, v0, m, full, kd);
    store_fixed32(fixed, cbytes, smbytes, v0, full, kd);
    const unsigned cnt = __popc(kd.e[0]) + __popc(kd.e[1]) + __popc(kd.e[2]) + __popc(kd.e[3]);
    if (speculative) {  // this thread's values, and those inside the window
      const unsigned mine = full ? 32u : (m > v0 ? min(m - v0, 32u) : 0u);
      spec_values += mine;
      spec_inside += mine - cnt;
    }

    unsigned base;
    const unsigned k = chunk_rank(cnt, &base, S.scan);  // [R]
    // The escape section: a list when 3k <= m, else a plane (the same in every coding thread).
    const bool plane = 3 * k > m;
    const unsigned esc_bytes = plane ? ((m + 15u) & ~15u) : ((3 * k + 15u) & ~15u);
    // The list's place in the ring: every coding thread works it out from its own copy of the
    // ring state and waits (bounded) for the room itself, so no barrier is needed before the
    // list is written.  A thread that gives up stops the CTA at [C].
    unsigned where, gap;
    ring_place(R.head, esc_bytes, kRingBytes, &where, &gap);
    if (tid == 0 && c != p.stall_chunk) st_relaxed_u64(&p.flags[c], kFlagAggregate | esc_bytes);  // publish early
    bool stop = failed || c == p.stall_chunk;  // (the stall test hook: this list is never resolved)
    if (!stop && !ring_room(S, R, gap, esc_bytes, p)) stop = true;
    R.made += gap + esc_bytes;
    R.head = where + esc_bytes;
    if (__any_sync(0xFFFFFFFFu, stop)) {
      // nothing to write: the CTA stops at [C]
    } else if (plane) {
      write_plane(S.xin[s], sw, smem_u32(S.ring) + where + v0, v0 < esc_bytes ? esc_bytes - v0 : 0u);
    } else {  // positions and exponents, in rank order
      // Each thread writes its own escapes; the exponent is read back from the staged input.
      // Shared memory is addressed with 32-bit shared-window addresses.
      const uint32_t esc = smem_u32(S.ring) + where;
      const uint32_t xs = smem_u32(S.xin[s]);  // value v0 + b at byte xs + (sw ^ (2b & 0x3E))
      unsigned m32 = 0;  // the flags compacted: value v0 + b at bit b
#pragma unroll
      for (int q = 0; q < 4; ++q) m32 |= compact8(kd.e[q]) << (8 * q);
      write_list32(m32, cnt, v0, base, k, esc, __reduce_max_sync(0xFFFFFFFFu, cnt) >= kDenseMin,
                   [&](unsigned b) { return lds_u16(xs + (sw ^ ((2 * b) & 0x3Eu))) >> 7; });
      if (tid < esc_bytes - 3 * k) sts_u8(esc + 3 * k + tid, 0);  // zero padding, < 16 bytes
    }
    if (bar_coders_or(stop)) break;  // [C] the list is complete in the ring; stage s is free again
    ++R.pushed;
    ++spec_chunks;
    if (tid == 0) {
      const unsigned qi = (R.pushed - 1) % kQueue;
      S.q_chunk[qi] = c;
      S.q_off[qi] = where;
      S.q_size[qi] = esc_bytes;
      S.q_gap[qi] = gap;
      __threadfence_block();
      S.q_pushed = R.pushed;
      // The next ticket was taken a chunk ago, so its round trip is already over; the one
      // after it is taken now and used a chunk later.
      S.ticket[s] = next_ticket;
      if (next_ticket < p.N) {
        issue_load(S, s, next_ticket, p, &in_map);
        pending |= 1u << s;
        next_ticket = atomicAdd(&p.ctrl->encode_ticket, 1u);
      }
    }
  }

  if (tid == 0) {
    __threadfence_block();
    S.coders_done = 1;  // the retiring warp drains the queue and leaves
    for (int s = 0; s < kStages; ++s)  // never leave a copy in flight
      if (pending & (1u << s)) {
        mbar_wait(&S.mbar[s], (parity >> s) & 1u, kWaitLimit);
        parity ^= 1u << s;
      }
    S.lb_parity = parity;
  }
  if (speculative && !skip)
    spec_verdict(S, p, e0, spec_acc, spec_nonfinite, spec_chunks, spec_fast, spec_values, spec_inside);
  if (p.values && !skip) {
    // Loopback: no chunk left to code, so decode.  The stages are free now, the ring once the
    // retiring warp has written out the last sections and left (bounded wait).
    if (tid == 0) {
      unsigned spins = 0, backoff = 64;
      S.dok = 1;
      while (S.retirer_done == 0) {
        if (read_status(p.status) != 0 || ++spins > p.spin_limit) {
          if (spins > p.spin_limit) set_error(p.status, ZC_ERR_TIMEOUT);
          S.dok = 0;
          break;
        }
        __nanosleep(backoff);
        backoff = backoff < 512 ? backoff * 2 : 512;
      }
      __threadfence_block();
    }
    bar_coders();
    if (S.dok)
      loopback_decode_slots(S, p.out, p.values, p.flags, p.ctrl, p.status, p.n, p.N, p.spin_limit, true);
  }
}

// n = 0: the raw form (32 bytes, the header alone) is shorter than the coded one (48 bytes).
__global__ void empty_stream_kernel(uint8_t* out, int base, Control* ctrl, unsigned long long* out_bytes) {
  unsigned long long* w = reinterpret_cast<unsigned long long*>(out);
  const int e0 = base >= 0 ? base : 0;  // no finite value: e0 = 0
  w[0] = kRawMagicWord | (static_cast<unsigned long long>(e0) << 56);
  w[1] = 0;
  w[2] = 0;
  w[3] = kHeaderBytes;
  ctrl->total = kHeaderBytes;
  if (out_bytes) *out_bytes = kHeaderBytes;
}

// After the encode kernel, as a programmatic dependent launch: when the coded stream is longer
// than the raw form, the stream becomes the raw form -- the header (byte 6 = 0, N = 0), the n
// values as they are (16-byte copies), zero padding -- and its length is reported again.
// Otherwise every CTA returns after one load.
constexpr int kRawThreads = 256;
constexpr int kRawVecPerThread = 4;

__global__ void __launch_bounds__(kRawThreads) raw_form_kernel(const uint16_t* in, uint64_t n, int base, uint8_t* out,
                                                               Control* ctrl, unsigned long long* out_bytes) {
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the encode kernel and its writes are done
  const unsigned long long raw = raw_stream_bytes(n);
  if (__ldcg(&ctrl->total) <= raw) return;
  const uint4* src = reinterpret_cast<const uint4*>(in);
  uint4* dst = reinterpret_cast<uint4*>(out + kHeaderBytes);
  const uint64_t nvec = n / 8;  // whole 16-byte vectors of values
  const uint64_t stride = static_cast<uint64_t>(gridDim.x) * kRawThreads;
  for (uint64_t i = static_cast<uint64_t>(blockIdx.x) * kRawThreads + threadIdx.x; i < nvec;
       i += stride * kRawVecPerThread) {
    uint4 v[kRawVecPerThread];
#pragma unroll
    for (int j = 0; j < kRawVecPerThread; ++j)
      if (i + j * stride < nvec) v[j] = __ldcs(src + i + j * stride);
#pragma unroll
    for (int j = 0; j < kRawVecPerThread; ++j)
      if (i + j * stride < nvec) __stcs(dst + i + j * stride, v[j]);
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    if (n % 8) {  // the last values and the zero padding: one 16-byte vector
      uint32_t w[4] = {0, 0, 0, 0};
      for (unsigned i = 0; i < n % 8; ++i) w[i >> 1] |= static_cast<uint32_t>(in[8 * nvec + i]) << (16 * (i & 1));
      dst[nvec] = make_uint4(w[0], w[1], w[2], w[3]);
    }
    const unsigned long long e0 = base >= 0 ? static_cast<unsigned>(base) : static_cast<unsigned>(__ldcg(&ctrl->e0));
    unsigned long long* hdr = reinterpret_cast<unsigned long long*>(out);
    hdr[0] = kRawMagicWord | (e0 << 56);
    hdr[1] = n;
    hdr[2] = 0;
    hdr[3] = raw;
    ctrl->total = raw;
    if (out_bytes) *out_bytes = raw;
  }
}

// Dynamic shared memory of the encode kernel: the layout plus room to align it to 1024 bytes.
constexpr int kEncodeSmemBytes = static_cast<int>(sizeof(EncodeSmem)) + 1024;
static_assert(kEncodeSmemBytes <= 233472 / kCtasPerSm - 1024, "kCtasPerSm CTAs fit an SM's shared memory");

// The driver's tensor-map encoder, looked up once through the runtime (so the library needs no
// link to the driver library).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    else
      cudaGetLastError();
  });
  return fn;
}

// The input's full chunks as a 3-D tensor of u16, {64, 64, n / 4096} (a chunk is 64 rows of 128
// bytes), one chunk per box, written to shared memory with the 128-byte swizzle.  With no full
// chunk the map is left zeroed and never used.
cudaError_t input_map(const uint16_t* in, uint64_t n, CUtensorMap* map) {
  std::memset(map, 0, sizeof *map);
  const uint64_t full = n / kChunk;
  if (full == 0) return cudaSuccess;
  const PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (encode == nullptr) return cudaErrorNotSupported;
  const cuuint64_t dims[3] = {64, 64, full};
  const cuuint64_t strides[2] = {128, 2 * kChunk};  // bytes, of dimensions 1 and 2
  const cuuint32_t box[3] = {64, 64, 1};
  const cuuint32_t unit[3] = {1, 1, 1};
  const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<uint16_t*>(in), dims, strides, box,
                            unit, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

cudaError_t encode_occupancy(int* per_sm) {
  const int smem = kEncodeSmemBytes;
  cudaError_t err = cudaFuncSetAttribute(encode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(per_sm, encode_kernel, kThreads, smem);
}

cudaError_t launch_encode(const uint16_t* in, uint64_t n, int base, uint8_t* out, unsigned long long* out_bytes,
                          uint8_t* ws, const DeviceInfo& dev, cudaStream_t stream, uint64_t stall_chunk,
                          unsigned spin_limit, uint16_t* loopback_values, int mode) {
  Control* ctrl = reinterpret_cast<Control*>(ws);
  if (n == 0) {
    empty_stream_kernel<<<1, 1, 0, stream>>>(out, base, ctrl, out_bytes);
    return cudaGetLastError();
  }
  EncodeParams p;
  p.in = in;
  p.n = n;
  p.N = num_chunks(n);
  p.out = out;
  p.ctrl = ctrl;
  p.flags = reinterpret_cast<unsigned long long*>(ws + kWsControlBytes + kWsPartialsBytes);
  p.out_bytes = out_bytes;
  p.base = base;
  p.status = dev.status;
  p.stall_chunk = stall_chunk;
  p.spin_limit = spin_limit;
  p.full_chunks = n / kChunk;
  p.values = loopback_values;
  p.mode = mode;
  CUtensorMap map;
  cudaError_t err = input_map(in, n, &map);
  if (err != cudaSuccess) return err;

  const int smem = kEncodeSmemBytes;
  const int per_sm = dev.encode_per_sm;
  uint64_t grid = static_cast<uint64_t>(per_sm > 0 ? per_sm : 1) * dev.sm_count;
  if (grid > p.N + 1) grid = p.N + 1;  // one CTA scans, the others code
  if (grid < 2) grid = 2;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  // After our own statistics kernel (auto mode): let this kernel start as that one finishes (it
  // reads e0 only after griddepcontrol.wait).  Not after a caller's kernel, which may still be
  // writing the input.
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = base < 0 && mode != kSpeculative ? 1 : 0;  // (the speculative launch follows the memset)
  TimingRecord t = timing_begin(mode == kGated ? ZC_KERNEL_REFIT_ENCODE : ZC_KERNEL_ENCODE, stream);
  err = cudaLaunchKernelEx(&cfg, encode_kernel, p, map);
  timing_end(t, stream);
  return err;
}

cudaError_t launch_raw_form(const uint16_t* in, uint64_t n, int base, uint8_t* out, unsigned long long* out_bytes,
                            uint8_t* ws, const DeviceInfo& dev, cudaStream_t stream) {
  if (n == 0) return cudaSuccess;  // the empty stream is written raw by the encode step
  const uint64_t nvec = n / 8;
  uint64_t grid = (nvec + kRawThreads * kRawVecPerThread - 1) / (kRawThreads * kRawVecPerThread);
  const uint64_t cap = 4ull * dev.sm_count;
  if (grid > cap) grid = cap;
  if (grid < 1) grid = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kRawThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // after our own encode kernel
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  TimingRecord t = timing_begin(ZC_KERNEL_RAW, stream);
  const cudaError_t err = cudaLaunchKernelEx(&cfg, raw_form_kernel, in, n, base, out,
                                             reinterpret_cast<Control*>(ws), out_bytes);
  timing_end(t, stream);
  return err;
}

// The speculative path, after the workspace is cleared: the encode kernel, speculating; then --
// each a programmatic dependent launch that returns at once unless the fallback word is set --
// the statistics kernel and the encode kernel again; then the raw-form step.
cudaError_t launch_speculative(const uint16_t* in, uint64_t n, uint8_t* out, unsigned long long* out_bytes,
                               uint8_t* ws, const DeviceInfo& dev, cudaStream_t stream, uint16_t* loopback_values) {
  cudaError_t err = launch_encode(in, n, ZC_BASE_AUTO, out, out_bytes, ws, dev, stream, ~uint64_t(0),
                                  kDefaultSpinLimit, loopback_values, kSpeculative);
  // (the loopback decodes the coded form: it never takes the raw pass, so no prediction)
  if (err == cudaSuccess) err = launch_stats(in, n, ws, dev, stream, loopback_values == nullptr, true);
  if (err == cudaSuccess)
    err = launch_encode(in, n, ZC_BASE_AUTO, out, out_bytes, ws, dev, stream, ~uint64_t(0), kDefaultSpinLimit,
                        loopback_values, kGated);
  if (err == cudaSuccess) err = launch_raw_form(in, n, ZC_BASE_AUTO, out, out_bytes, ws, dev, stream);
  return err;
}

}  // namespace zc
