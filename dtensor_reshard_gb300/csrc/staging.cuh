// staging.cuh -- pieces shared by the shared-memory staged kernels (sm_103a):
// mbarrier waits with a poll limit, cp.async.bulk copies, a byte funnel, and
// the walk of a CTA's work units in stage-sized chunks.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"

namespace rs {
namespace staging {

// try_wait polls before a wait is declared lost (a poll may suspend the thread
// for a short, hardware-defined time: this is of the order of a second).
constexpr uint32_t kWaitPolls = 1u << 22;

enum : unsigned int {
  kStatusProducerWait = 1,  // producer gave up waiting for a free stage
  kStatusConsumerWait = 2,  // consumer gave up waiting for a loaded stage
  kStatusSelfTest = 3,      // the self-test's deliberately unanswered wait ran out
  kStatusTransposeAlign = 4  // a transpose block did not allow its launch's element width
};

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count));
}
__device__ __forceinline__ void mbar_arrive_expect(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
// Wait for the phase with the given parity to complete; false after `polls` polls.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t polls) {
  for (uint32_t i = 0; i < polls; ++i) {
    uint32_t done;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; "
        "selp.u32 %0, 1, 0, p; }"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}
__device__ __forceinline__ void bulk_load(void* sdst, const void* gsrc, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_addr(sdst)),
      "l"(gsrc), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}
__device__ __forceinline__ void bulk_store(void* gdst, const void* ssrc, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst),
               "r"(smem_addr(ssrc)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read_all_but_newest() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// 16 bytes global -> shared through the load/store unit (L2 only); both
// addresses 16-byte aligned.
__device__ __forceinline__ void cp_async16(void* sdst, const void* gsrc) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(sdst)), "l"(gsrc)
               : "memory");
}
// The mbarrier's current phase also waits for this thread's cp.async copies
// issued so far (its pending count goes up now and down when they land).
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Bytes [o, o + 16) of the 32 bytes A:B, with q = o / 4 and
// sel = 0x3210 + 0x1111 * (o % 4) (byte-permute selector).
__device__ __forceinline__ uint4 funnel16(const uint4& A, const uint4& B, uint32_t q,
                                          uint32_t sel) {
  const uint32_t x0 = q == 0 ? A.x : q == 1 ? A.y : q == 2 ? A.z : A.w;
  const uint32_t x1 = q == 0 ? A.y : q == 1 ? A.z : q == 2 ? A.w : B.x;
  const uint32_t x2 = q == 0 ? A.z : q == 1 ? A.w : q == 2 ? B.x : B.y;
  const uint32_t x3 = q == 0 ? A.w : q == 1 ? B.x : q == 2 ? B.y : B.z;
  const uint32_t x4 = q == 0 ? B.x : q == 1 ? B.y : q == 2 ? B.z : B.w;
  return make_uint4(__byte_perm(x0, x1, sel), __byte_perm(x1, x2, sel), __byte_perm(x2, x3, sel),
                    __byte_perm(x3, x4, sel));
}

// n / div for n < 2^32 by multiply and shift (Granlund-Montgomery).
struct FastDiv32 {
  uint32_t m, l;
  __device__ __forceinline__ explicit FastDiv32(uint32_t div) {
    l = 0;
    while ((uint64_t(1) << l) < div) ++l;
    m = uint32_t(((uint64_t(1) << 32) * ((uint64_t(1) << l) - div)) / div + 1);
  }
  __device__ __forceinline__ uint32_t div(uint32_t n) const {
    return uint32_t((uint64_t(__umulhi(n, m)) + n) >> l);
  }
};

__device__ __forceinline__ uint32_t word_at(const uint4& v, uint32_t i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// Bytes [lo, hi) of the 16-byte granule v to the 16-byte aligned address g,
// in the widest naturally aligned stores that fit.
__device__ __forceinline__ void store_partial16(unsigned char* g, const uint4& v, uint32_t lo,
                                                uint32_t hi) {
  while (lo < hi) {
    const uint32_t w = word_at(v, lo >> 2);
    if ((lo & 7u) == 0 && lo + 8 <= hi) {
      *reinterpret_cast<uint2*>(g + lo) = make_uint2(w, word_at(v, (lo >> 2) + 1));
      lo += 8;
    } else if ((lo & 3u) == 0 && lo + 4 <= hi) {
      *reinterpret_cast<uint32_t*>(g + lo) = w;
      lo += 4;
    } else if ((lo & 1u) == 0 && lo + 2 <= hi) {
      *reinterpret_cast<uint16_t*>(g + lo) = uint16_t(w >> (8u * (lo & 3u)));
      lo += 2;
    } else {
      g[lo] = uint8_t(w >> (8u * (lo & 3u)));
      lo += 1;
    }
  }
}

// The destination bytes [lo, hi) that granule k of a row of n bytes covers,
// G = the row's granule count.
__device__ __forceinline__ void granule_span(uint32_t dmis, uint32_t n, uint32_t G, uint32_t k,
                                             uint32_t* lo, uint32_t* hi) {
  *lo = k == 0 ? dmis : 0u;
  *hi = k + 1 == G ? ((dmis + n - 1u) & 15u) + 1u : 16u;
}

// One chunk: at most one stage's worth of one tile.
struct Chunk {
  int ti;
  uint32_t kind;   // 0: bytes [a, b) of a run; 1: whole rows [a, b); 2: bytes [b, b+bytes) of row a
  int64_t a, b;
  uint32_t bytes;  // bytes of the tile the chunk covers
};

// One chunk, handed from the producer to its consumers together with its stage
// (when CTAs take their work from a queue rather than a fixed range).
struct StageDesc {
  int32_t ti;  // tile index; -1: no more chunks
  uint32_t kind, bytes;
  int64_t a, b;
};

// The next piece of a launch's work queue {next piece, CTAs finished}, one per
// call of the warp (lane 0 asks, every lane gets the answer).
__device__ __forceinline__ uint32_t grab_piece(unsigned int* queue, int lane) {
  uint32_t piece = 0;
  if (lane == 0) piece = atomicAdd(&queue[0], 1u);
  return __shfl_sync(0xffffffffu, piece, 0);
}

// After every warp of the CTA is done: count the CTA out of the launch; the
// last one puts the launch's queue slot back to zero for the next launch.
__device__ __forceinline__ void finish_queue(unsigned int* queue) {
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(&queue[1], 1u) == gridDim.x - 1) {
      atomicExch(&queue[0], 0u);
      atomicExch(&queue[1], 0u);
    }
  }
}

// Walks the chunks of this CTA's unit range (the same equal split of the
// program's work units as the vector kernel); the producer and the consumers
// each run their own copy and see the same sequence.  A stage holds STAGE
// bytes.  PAD = 0: rows are packed back to back and pieces are STAGE bytes.
// PAD > 0: pieces of runs and long rows are STAGE - PAD bytes and a row that
// is not source-contiguous with its neighbours takes a slot of
// round16(row_bytes + PAD) bytes (room for realignment slack).
template <uint32_t STAGE, uint32_t PAD>
struct ChunkWalker {
  static constexpr uint32_t kPiece = STAGE - PAD;
  static_assert(kPiece % 16 == 0, "pieces must keep 16-byte granularity");
  // Most rows in one chunk when PAD > 0 (a row table entry each).
  static constexpr uint32_t kMaxRows = STAGE / ((1u + PAD + 15u) & ~15u);

  const KernelParams* p = nullptr;
  int64_t u0 = 0, u1 = 0;
  int ti = 0;
  int64_t pos, end;
  uint32_t kind, per;  // per: rows per chunk (kind 1) or pieces per row (kind 2)
  reshard_tile_t t;
  bool live;
  bool live_once = false;  // start_range has run before (ti is meaningful)

  __device__ __forceinline__ static uint32_t slot(uint32_t row_bytes) {
    return PAD == 0 ? row_bytes : (row_bytes + PAD + 15u) & ~15u;
  }
  // Consecutive rows of the tile follow one another in the source buffer.
  __device__ __forceinline__ static bool source_contiguous(const reshard_tile_t& t) {
    return t.src_row_stride == int64_t(t.row_bytes) &&
           (t.nplanes == 1 || t.src_plane_stride == int64_t(t.nrows) * t.row_bytes);
  }
  // Bytes a row of n bytes takes in an output stage: the 16-byte granules its
  // destination range touches, whatever its alignment.
  __device__ __forceinline__ static uint32_t out_stride(uint32_t n) { return (n + 30u) & ~15u; }
  // Whole rows per chunk; 0 when a row has to be split into pieces.  PAD = 0:
  // rows back to back.  PAD > 0: a source-contiguous run of rows shares one
  // piece, other rows take a slot each; either way the rows' output granules
  // fit in one stage and the row table.
  __device__ __forceinline__ static uint32_t rows_per_chunk(const reshard_tile_t& t) {
    if (PAD == 0) return t.row_bytes <= STAGE ? STAGE / t.row_bytes : 0u;
    if (slot(t.row_bytes) > STAGE && (!source_contiguous(t) || t.row_bytes > kPiece)) return 0u;
    uint32_t per = source_contiguous(t) ? kPiece / t.row_bytes : STAGE / slot(t.row_bytes);
    per = min(per, STAGE / out_stride(t.row_bytes));
    return min(per, kMaxRows);
  }

  __device__ void enter_tile() {
    t = p->tiles[ti];
    const int64_t tb = p->prefix[ti], te = p->prefix[ti + 1];
    const int64_t a = u0 - tb, b = (u1 < te ? u1 : te) - tb;
    if (t.nrows == 1 && t.nplanes == 1) {
      kind = 0;
      pos = a * kUnitBytes;
      end = min(b * kUnitBytes, int64_t(t.row_bytes));
      return;
    }
    const int64_t upr = rows_per_unit(t.row_bytes);
    const int64_t rows = int64_t(t.nrows) * t.nplanes;
    const int64_t r0 = a * upr, r1 = min(b * upr, rows);
    const uint32_t rpc = rows_per_chunk(t);
    if (rpc > 0) {
      kind = 1;
      per = rpc;
      pos = r0;
      end = r1;
    } else {
      kind = 2;
      per = (t.row_bytes + kPiece - 1) / kPiece;
      pos = r0 * per;
      end = r1 * per;
    }
  }
  __device__ void start(const KernelParams* kp) {
    p = kp;
    u0 = kp->total_units * int64_t(blockIdx.x) / int64_t(gridDim.x);
    u1 = kp->total_units * int64_t(blockIdx.x + 1) / int64_t(gridDim.x);
    live = u0 < u1;
    if (!live) return;
    int lo = 0, hi = kp->ntiles - 1;  // largest tile with prefix <= u0
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (kp->prefix[mid] <= u0) lo = mid;
      else hi = mid - 1;
    }
    ti = lo;
    enter_tile();
  }
  // Walk units [a, b) instead of the CTA's equal share (a piece handed out at
  // run time); the tile search starts at the current tile when the piece lies
  // ahead of it, as pieces of one CTA do.  Called by all 32 lanes of a warp at
  // once (a producer warp, whose lanes run the walk in step): each round the
  // lanes test 32 evenly spaced tiles and a ballot keeps the stretch between
  // the last one at or before u0 and the next, so a program of 4096 tiles takes
  // 3 rounds of loads from the prefix table instead of 12 dependent ones.
  __device__ void start_range(const KernelParams* kp, int64_t a, int64_t b) {
    const bool ahead = live_once && p == kp && a >= kp->prefix[ti];
    p = kp;
    u0 = a;
    u1 = b;
    live = u0 < u1;
    live_once = true;
    if (!live) return;
    const int lane = int(threadIdx.x & 31u);
    int lo = ahead ? ti : 0, hi = kp->ntiles - 1;  // largest tile with prefix <= u0
    while (lo < hi) {  // prefix[lo] <= u0 throughout
      const int step = (hi - lo + 31) / 32;
      const int at = lo + (lane + 1) * step;
      const unsigned le = __ballot_sync(0xffffffffu, at <= hi && kp->prefix[at] <= u0);
      if (le != 0u) lo += (32 - __clz(int(le))) * step;  // the last sample at or before u0
      hi = min(hi, lo + step - 1);
    }
    ti = lo;
    enter_tile();
  }
  __device__ bool next(Chunk* c) {
    while (live && pos >= end) {
      const int64_t te = p->prefix[ti + 1];
      if (te >= u1) {
        live = false;
        break;
      }
      u0 = te;
      ++ti;
      enter_tile();
    }
    if (!live) return false;
    c->ti = ti;
    c->kind = kind;
    if (kind == 0) {
      const int64_t e = min(end, pos + int64_t(kPiece));
      c->a = pos;
      c->b = e;
      c->bytes = uint32_t(e - pos);
      pos = e;
    } else if (kind == 1) {
      const int64_t e = min(end, pos + int64_t(per));
      c->a = pos;
      c->b = e;
      c->bytes = uint32_t((e - pos) * t.row_bytes);
      pos = e;
    } else {
      const int64_t row = pos / per, piece = pos - row * per;
      const int64_t b0 = piece * kPiece;
      const int64_t b1 = min(int64_t(t.row_bytes), b0 + int64_t(kPiece));
      c->a = row;
      c->b = b0;
      c->bytes = uint32_t(b1 - b0);
      pos += 1;
    }
    return true;
  }
};

__device__ __forceinline__ int64_t src_row(const reshard_tile_t& t, int64_t r) {
  if (t.nplanes == 1) return t.src_off + r * t.src_row_stride;
  const int64_t pl = r / t.nrows, q = r - pl * t.nrows;
  return t.src_off + pl * t.src_plane_stride + q * t.src_row_stride;
}
__device__ __forceinline__ int64_t dst_row(const reshard_tile_t& t, int64_t r) {
  if (t.nplanes == 1) return t.dst_off + r * t.dst_row_stride;
  const int64_t pl = r / t.nrows, q = r - pl * t.nrows;
  return t.dst_off + pl * t.dst_plane_stride + q * t.dst_row_stride;
}

}  // namespace staging
}  // namespace rs
