// transpose.cu -- transpose blocks: narrow innermost pieces regrouped by rows (sm_103a).
//
// A block covers nrows consecutive rows of row_bytes on the wide side (one
// contiguous range of one buffer, or of every buffer of one destination group)
// and seg_count narrow segments, each a dense nrows x width range of its own
// buffer (or destination group) that fills bytes [col, col + width) of every
// wide row.  A CTA takes a contiguous share of the program's blocks and, per
// block:
//   gather  (narrow sources -> wide destination group): every thread loads
//           whole aligned 16-byte granules of the segments' dense ranges and
//           puts their elements into their columns of a shared-memory image of
//           the rows, then the image goes out with 16-byte stores to every
//           replica;
//   scatter (wide source -> narrow destination groups): the rows come in with
//           16-byte loads, then every thread builds whole aligned 16-byte
//           granules of the segments' dense ranges from the image and stores
//           each to every replica of its segment.
// The shared-memory image is shifted by the wide side's address mod 16, so its
// 16-byte vectors line up with aligned global addresses.  Inside a granule the
// elements are U bytes (the widest unit every address, width and column of the
// block allows) and follow a segment's rows in order, so a thread finds the
// image position of its first element with one division and steps from there;
// the granules of all segments are numbered in one sequence, so every thread
// has the same amount of work whatever the segments' sizes.
#include <cuda_runtime.h>

#include <cstdint>
#include <map>
#include <mutex>
#include <string>

#include "internal.h"
#include "staging.cuh"

namespace rs {
namespace {

constexpr int kTThreads = 256;
constexpr int kTVecUnroll = 4;  // wide-side 16-byte loads in flight per thread
constexpr int kImageBytes = int(kTransposeBlockBytes) + 64;
// DB (programs with scatter blocks): two images, a scatter block's wide rows
// bulk-loaded into one while the previous scatter block is built from the other.
// Programs of gather blocks only keep one image (the second one's shared memory
// was measured to cost them 5-10%).
template <bool DB> constexpr int dyn_smem() { return DB ? 2 * kImageBytes : kImageBytes; }
constexpr int kMaxReplicaPtrs = int(kTransposeMaxReplicaPtrs);

struct TransposeParams {
  unsigned int* status;
  const reshard_tblock_t* blocks;
  const reshard_tseg_t* segs;
  const uint32_t* goff;
  const uint16_t* gbuf;
  int64_t nblocks;
  int32_t nbufs;
  uint32_t flags;
  unsigned char* bufs[RESHARD_MAX_EXEC_BUFFERS];
};

// Division by a runtime-invariant divisor (Granlund and Montgomery, PLDI 1994,
// round-up method): n / d = (umulhi(n, m) + n) >> l for every 32-bit n.
__device__ __forceinline__ void fastdiv_init(uint32_t d, uint32_t* m, uint32_t* l) {
  uint32_t s = 0;
  while ((uint64_t(1) << s) < d) ++s;
  *l = s;
  *m = uint32_t(((uint64_t(1) << 32) * ((uint64_t(1) << s) - d)) / d + 1);
}
__device__ __forceinline__ uint32_t fastdiv(uint32_t n, uint32_t m, uint32_t l) {
  return uint32_t((uint64_t(__umulhi(n, m)) + n) >> l);
}

struct SegInfo {
  const unsigned char* src;  // gather: narrow source at the block's row 0
  int64_t off;               // scatter: narrow byte offset at the block's row 0
  uint32_t units;            // width / U
  uint32_t col;              // byte column inside a wide row
  uint32_t m, l;             // fast division by units
  uint32_t rbeg, rcnt;       // scatter: replica pointers [rbeg, rbeg + rcnt) of ptrs[]
  uint32_t gstart;           // first granule of the segment
  uint32_t gmis;             // narrow global address mod 16 (replica 0 for scatter)
  uint32_t nbytes;           // width * nrows
  uint32_t moved;            // gmis differs from the block the granule plans were made for
};

template <int U> struct UType;
template <> struct UType<1> { using T = uint8_t; };
template <> struct UType<2> { using T = uint16_t; };
template <> struct UType<4> { using T = uint32_t; };
template <> struct UType<8> { using T = uint2; };

// segment owning granule g (largest k with gstart[k] <= g)
__device__ __forceinline__ int find_granule(const SegInfo* si, int K, uint32_t g) {
  int lo = 0, hi = K - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (si[mid].gstart <= g) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// Element i (of 16 / U) of a 16-byte granule held as four words.
template <int U>
__device__ __forceinline__ typename UType<U>::T granule_elem(const uint4& v, int i) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  if constexpr (U == 8) {
    return make_uint2(w[2 * i], w[2 * i + 1]);
  } else if constexpr (U == 4) {
    return w[i];
  } else if constexpr (U == 2) {
    return uint16_t(w[i >> 1] >> (16 * (i & 1)));
  } else {
    return uint8_t(w[i >> 2] >> (8 * (i & 3)));
  }
}
template <int U>
__device__ __forceinline__ void granule_put(uint32_t (&w)[4], int i, typename UType<U>::T e) {
  if constexpr (U == 8) {
    w[2 * i] = e.x;
    w[2 * i + 1] = e.y;
  } else if constexpr (U == 4) {
    w[i] = e;
  } else if constexpr (U == 2) {
    w[i >> 1] |= uint32_t(e) << (16 * (i & 1));
  } else {
    w[i >> 2] |= uint32_t(e) << (8 * (i & 3));
  }
}

// The plan of one granule: which segment it belongs to, which of its bytes
// [lo, hi) are the segment's, the image byte of its first element (counted
// from the image's shifted origin) and, for the general walk, that element's
// column in its row.  Granules come in three kinds:
//   ROWS  a whole granule of 16 / width whole rows (width divides 16 and the
//         narrow start's offset mod 16): element i is at row i / units,
//         column i % units, a pattern the compiler unrolls;
//   INROW a whole granule of 16 bytes inside one row (16 divides the width,
//         the narrow range 16-byte aligned): one unaligned 16-byte stretch of
//         the image;
//   WALK  anything else: elements in order, wrapping to the next row.
// A plan depends on the block's shape and on the narrow ranges' addresses mod
// 16 only, so a CTA keeps its threads' plans over blocks of the same shape and
// redoes only those of segments whose narrow address mod 16 moved.
constexpr uint32_t kKindNone = 0, kKindWalk = 1, kKindRows = 2, kKindInrow = 3;
constexpr int kSlots = 6;  // planned granules per thread (more are walked each block)

// One 32-bit word per planned granule: image byte of the first element (before
// the image shift, below 2^15), segment, kind, and the first element's column.
// The granule's bytes [lo, hi) follow from its segment and index.
__device__ __forceinline__ uint32_t plan_off(uint32_t m) { return m & 0x7fffu; }
__device__ __forceinline__ uint32_t plan_k(uint32_t m) { return (m >> 15) & 0x7fu; }
__device__ __forceinline__ uint32_t plan_kind(uint32_t m) { return (m >> 22) & 0x3u; }
__device__ __forceinline__ uint32_t plan_c(uint32_t m) { return m >> 24; }
static_assert(kTransposeBlockBytes < (1 << 15) && kTransposeMaxSegs <= 128 &&
                  kTransposeMaxWidth <= 129, "granule plan fields");

// Bytes [lo, hi) of granule j that belong to its segment (hi <= lo: none).
__device__ __forceinline__ void granule_span(const SegInfo& s, uint32_t j, uint32_t* lo,
                                             uint32_t* hi) {
  *lo = j == 0 ? s.gmis : 0u;
  const int32_t h = int32_t(s.gmis + s.nbytes) - int32_t(16u * j);
  *hi = h >= 16 ? 16u : (h > 0 ? uint32_t(h) : 0u);
}

// Does the segment's whole granules take a fast kind (ROWS or INROW)?
template <int U>
__device__ __forceinline__ bool fast_segment(const SegInfo& s) {
  const uint32_t width = s.units * U;
  return (16u % width == 0 && s.gmis % width == 0) || (width % 16u == 0 && s.gmis == 0);
}

// Partial granule e of a block (e < 2 K): the first (e even) or the last (e odd)
// granule of segment e / 2, when that granule is not whole and the segment's
// whole granules take a fast kind; false otherwise.
template <int U>
__device__ __forceinline__ bool edge_granule(const SegInfo* si, uint32_t e, uint32_t* k,
                                             uint32_t* j) {
  const SegInfo& s = si[e >> 1];
  if (!fast_segment<U>(s)) return false;
  const uint32_t n = (s.gmis + s.nbytes + 15u) >> 4;  // granules of the segment
  if (n == 0) return false;
  *k = e >> 1;
  if ((e & 1u) == 0) {
    *j = 0;
    return s.gmis != 0 || s.nbytes < 16;  // the first granule, when not whole
  }
  *j = n - 1;
  return n > 1 && ((s.gmis + s.nbytes) & 15u) != 0;  // the last one, when not whole
}

// Plan of granule j of segment k.  With EDGE false, a granule that is not
// whole (the first or last of a segment whose narrow range is not 16-byte
// aligned at that end) of a segment whose whole granules take a fast kind is
// left out (kind none): the edge pass takes those, so that warps of whole
// granules do not also run the partial-granule path.
template <int U, bool EDGE = false>
__device__ __forceinline__ uint32_t plan_of(const SegInfo& s, uint32_t k, uint32_t j, uint32_t L) {
  uint32_t lo, hi;
  granule_span(s, j, &lo, &hi);
  if (hi <= lo || (!EDGE && (lo != 0 || hi != 16) && fast_segment<U>(s)))
    return k << 15;  // kind none
  const uint32_t e0 = (16u * j + lo - s.gmis) / U;
  const uint32_t row = fastdiv(e0, s.m, s.l);
  const uint32_t c = e0 - row * s.units;
  const uint32_t off = s.col + row * L + c * U;
  uint32_t kind = kKindWalk;
  const uint32_t width = s.units * U;
  if (lo == 0 && hi == 16) {
    // a whole granule starts at a row boundary when the width divides 16 and the
    // narrow start's offset mod 16; it lies inside one row when 16 divides the
    // width and the narrow start is aligned
    if (16u % width == 0 && s.gmis % width == 0) kind = kKindRows;
    else if (width % 16u == 0 && s.gmis == 0) kind = kKindInrow;
  }
  return off | (k << 15) | (kind << 22) | (c << 24);
}

// A whole granule of rows: element i at row i / UNITS, column i % UNITS.
template <int U, int UNITS, bool GATHER>
__device__ __forceinline__ void rows_move(unsigned char* img_at, uint32_t L, uint32_t (&words)[4],
                                          const uint4& v) {
  using T = typename UType<U>::T;
  constexpr int E = 16 / U;
#pragma unroll
  for (int i = 0; i < E; ++i) {
    unsigned char* a = img_at + (i / UNITS) * L + (i % UNITS) * U;
    if constexpr (GATHER) *reinterpret_cast<T*>(a) = granule_elem<U>(v, i);
    else granule_put<U>(words, i, *reinterpret_cast<const T*>(a));
  }
}
template <int U, bool GATHER>
__device__ __forceinline__ void rows_dispatch(uint32_t units, unsigned char* img_at, uint32_t L,
                                              uint32_t (&words)[4], const uint4& v) {
  constexpr int E = 16 / U;
  switch (units) {
    case 1: rows_move<U, 1, GATHER>(img_at, L, words, v); break;
    case 2: if constexpr (E >= 2) rows_move<U, 2, GATHER>(img_at, L, words, v); break;
    case 4: if constexpr (E >= 4) rows_move<U, 4, GATHER>(img_at, L, words, v); break;
    case 8: if constexpr (E >= 8) rows_move<U, 8, GATHER>(img_at, L, words, v); break;
    default: if constexpr (E >= 16) rows_move<U, 16, GATHER>(img_at, L, words, v); break;
  }
}

// The elements [lo, hi) of a granule in order, wrapping from the end of a row to
// the start of the next one (c: column of the first element in its row).
template <int U, bool GATHER>
__device__ __forceinline__ void walk_move(unsigned char* to, uint32_t units, uint32_t wrap,
                                          uint32_t c, uint32_t lo, uint32_t hi,
                                          uint32_t (&words)[4], const uint4& v) {
  using T = typename UType<U>::T;
  constexpr int E = 16 / U;
  const int ilo = int(lo / U), ihi = int(hi / U);
#pragma unroll
  for (int i = 0; i < E; ++i) {
    if (i >= ilo && i < ihi) {
      if constexpr (GATHER) *reinterpret_cast<T*>(to) = granule_elem<U>(v, i);
      else granule_put<U>(words, i, *reinterpret_cast<const T*>(to));
      to += U;
      if (++c == units) {
        c = 0;
        to += wrap;
      }
    }
  }
}

// The image bytes of one granule (scatter: into words; gather: from v).
template <int U, bool GATHER>
__device__ __forceinline__ void granule_move(const SegInfo& s, uint32_t meta, uint32_t lo,
                                             uint32_t hi, unsigned char* img_at, uint32_t L,
                                             uint32_t (&words)[4], const uint4& v) {
  const uint32_t kind = plan_kind(meta);
  if (kind == kKindRows) {
    rows_dispatch<U, GATHER>(s.units, img_at, L, words, v);
  } else if (kind == kKindInrow) {
    if constexpr (GATHER) {
      using T = typename UType<U>::T;
#pragma unroll
      for (int i = 0; i < 16 / U; ++i) *reinterpret_cast<T*>(img_at + i * U) = granule_elem<U>(v, i);
    } else {
      // 16 bytes at any alignment: five aligned 4-byte words funnel-shifted by the
      // byte offset (the reads stay inside the image and its slack)
      const uint32_t a = uint32_t(reinterpret_cast<uintptr_t>(img_at) & 3u);
      const uint32_t* w = reinterpret_cast<const uint32_t*>(img_at - a);
      const uint32_t sh = 8u * a;
      const uint32_t w0 = w[0], w1 = w[1], w2 = w[2], w3 = w[3], w4 = sh ? w[4] : 0u;
      words[0] = __funnelshift_r(w0, w1, sh);
      words[1] = __funnelshift_r(w1, w2, sh);
      words[2] = __funnelshift_r(w2, w3, sh);
      words[3] = __funnelshift_r(w3, w4, sh);
    }
  } else {
    walk_move<U, GATHER>(img_at, s.units, L - s.units * U, plan_c(meta), lo, hi, words, v);
  }
}

// A bulk copy shared -> global whose lines L2 evicts first: a gather's image goes
// out once to each replica and is not read again, while the narrow source's
// boundary granules are read again by the next block (with the normal policy the
// image stores displaced them: reads of the 12-replica gather rose from 1.07 to
// 1.39 times its source bytes).
__device__ __forceinline__ void bulk_store_evict_first(void* gdst, const void* ssrc,
                                                       uint32_t bytes) {
  asm volatile(
      "{ .reg .b64 pol; createpolicy.fractional.L2::evict_first.b64 pol, 1.0; "
      "cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, pol; }" ::"l"(
          gdst),
      "r"(staging::smem_addr(ssrc)), "r"(bytes)
      : "memory");
}

// every bulk copy this thread committed has finished reading shared memory
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// gather: an aligned 16-byte granule of a narrow source range, with the normal
// cache policy.  A block's range shares its first and last 32-byte sectors with
// the neighbouring blocks' ranges; evict-first loads dropped those sectors before
// the neighbour read its half, and the narrow side was read from DRAM 1.5 times
// (a gather of 58-byte pieces into 12 replicas).
__device__ __forceinline__ uint4 narrow_load(const unsigned char* p) {
  return *reinterpret_cast<const uint4*>(p);
}

// scatter: a granule built from the image goes to every replica of its segment.
__device__ __forceinline__ void scatter_store(const SegInfo& s, uint32_t j, uint32_t lo,
                                              uint32_t hi, const uint32_t (&words)[4],
                                              unsigned char* const* ptrs) {
  const uint4 v = make_uint4(words[0], words[1], words[2], words[3]);
  for (uint32_t r = 0; r < s.rcnt; ++r) {
    unsigned char* base = ptrs[s.rbeg + r] + s.off;  // segment byte 0 of this replica
    if ((reinterpret_cast<uintptr_t>(base) & 15u) == s.gmis) {
      // aligned like replica 0: a whole granule in one store, a partial one in the
      // widest aligned stores that fit
      unsigned char* gp = base - s.gmis + 16 * size_t(j);
      if (lo == 0 && hi == 16) __stcs(reinterpret_cast<uint4*>(gp), v);
      else staging::store_partial16(gp, v, lo, hi);
    } else {
      for (uint32_t b = lo; b < hi; ++b)
        base[16 * j + b - s.gmis] = uint8_t(staging::word_at(v, b >> 2) >> (8u * (b & 3u)));
    }
  }
}

// U: the element width in bytes (1, 2, 4 or 8) that divides every block's row
// length, columns, widths and narrow addresses (the host takes it from the
// plan's offsets and the buffers' addresses); a block that does not allow it
// is skipped and reported in the status word.
template <int U, bool DB>
__global__ void __launch_bounds__(kTThreads, 4)
    reshard_transpose_kernel(const __grid_constant__ TransposeParams p) {
  extern __shared__ __align__(16) unsigned char dyn[];
  // wide rows, shifted by the wide address mod 16: gathers build theirs in image 0,
  // scatter blocks alternate between images 0 and 1
  __shared__ SegInfo si[kTransposeMaxSegs];
  __shared__ unsigned char* ptrs[kMaxReplicaPtrs];
  __shared__ unsigned int s_align;
  __shared__ uint32_t s_ngran;
  __shared__ __align__(8) uint64_t s_bar[2];  // one bulk load in flight per image
  const bool congruent = (p.flags & kFlagDstCongruent) != 0;
  const int64_t b0 = p.nblocks * int64_t(blockIdx.x) / int64_t(gridDim.x);
  const int64_t b1 = p.nblocks * int64_t(blockIdx.x + 1) / int64_t(gridDim.x);
  if (DB && threadIdx.x == 0) {
    staging::mbar_init(&s_bar[0], 1);
    staging::mbar_init(&s_bar[1], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // The wide rows of scatter block b -> image `buf` by one bulk copy of the aligned
  // 16-byte granules holding them (thread 0; at most kTransposeBlockBytes + 16
  // bytes, inside the image).
  auto load_wide = [&](int64_t b, uint32_t buf) {
    const reshard_tblock_t nb = p.blocks[b];
    const unsigned char* src = p.bufs[nb.wide] + nb.wide_off;
    const uint32_t m = uint32_t(reinterpret_cast<uintptr_t>(src) & 15u);
    const uint32_t bytes = (m + nb.row_bytes * nb.nrows + 15u) & ~15u;
    staging::mbar_arrive_expect(&s_bar[buf], bytes);
    staging::bulk_load(dyn + buf * kImageBytes, src - m, bytes, &s_bar[buf]);
  };
  // this thread's granules tid + s * kTThreads, planned for the current shape
  uint32_t plan[kSlots];
  // uniform over the CTA: scatter blocks seen, loads issued per image, wait parities
  uint32_t nscatter = 0, pending = 0, parity = 0;
  bool have_plan = false;
  int R = 0;  // gather: replicas of the wide destination group (in ptrs[0..R))
  for (int64_t bi = b0; bi < b1; ++bi) {
    const reshard_tblock_t blk = p.blocks[bi];
    const uint32_t L = blk.row_bytes, nr = blk.nrows, K = blk.seg_count;
    const uint32_t n = L * nr;
    const bool gather = blk.direction == 0;
    // the shape of the previous block of this CTA: plans, segment layout and
    // replica pointers stay, only the offsets move
    const bool same = have_plan && (blk.flags & RESHARD_TBLOCK_SAME_SHAPE) != 0;
    // ... and its rows and narrow ranges follow the previous block's: every offset
    // advances by rows x width, with no segment record to read and no alignment to
    // check again (the advances are multiples of the element width)
    const bool follows = same && (blk.flags & RESHARD_TBLOCK_FOLLOWS) != 0;
    // the previous gather block's bulk stores have read its image (thread 0 issued them)
    if (threadIdx.x == 0) bulk_wait_read_all();
    __syncthreads();  // the previous block is completely done with its image, si and ptrs
    const uint32_t buf = (DB && !gather) ? (nscatter & 1u) : 0u;
    unsigned char* img = dyn + buf * kImageBytes;
    if (DB && !gather) {
      // this block's rows (unless already on their way), then the next scatter
      // block's into the other image, which the previous block is done with
      if (!((pending >> buf) & 1u)) {
        if (threadIdx.x == 0) load_wide(bi, buf);
        pending |= 1u << buf;
      }
      if (bi + 1 < b1 && p.blocks[bi + 1].direction != 0) {
        if (threadIdx.x == 0) load_wide(bi + 1, buf ^ 1u);
        pending |= 1u << (buf ^ 1u);
      }
    }
    // wide-side pointers: gather -> the destination group in ptrs[0..R); scatter -> source
    const unsigned char* wsrc = nullptr;
    if (gather) {
      if (!same) {  // (a block of the same shape has the same destination group)
        const uint32_t g0 = p.goff[blk.wide];
        R = int(p.goff[blk.wide + 1] - g0);
        for (int i = threadIdx.x; i < R; i += kTThreads) ptrs[i] = p.bufs[p.gbuf[g0 + i]];
      }
    } else {
      wsrc = p.bufs[blk.wide] + blk.wide_off;
    }
    if (follows) {
      for (uint32_t k = threadIdx.x; k < K; k += kTThreads) {
        const uint32_t adv = si[k].nbytes;  // rows x width
        if (gather) si[k].src += adv;
        else si[k].off += adv;
        const uint32_t gm = (si[k].gmis + adv) & 15u;
        si[k].moved = si[k].moved | (gm != si[k].gmis ? 1u : 0u);
        si[k].gmis = gm;
      }
    } else {
      if (threadIdx.x == 0) s_align = L;
    }
    __syncthreads();
    const uint32_t mis = gather ? uint32_t(reinterpret_cast<uintptr_t>(ptrs[0] + blk.wide_off) & 15u)
                                : uint32_t(reinterpret_cast<uintptr_t>(wsrc) & 15u);
    // per-segment set-up (one thread per segment), alignment of every narrow access
    for (uint32_t k = threadIdx.x; k < K && !follows; k += kTThreads) {
      const reshard_tseg_t sg = p.segs[blk.seg_begin + k];
      unsigned int a = sg.width | (mis + sg.col);
      uint32_t gm;
      if (gather) {
        si[k].src = p.bufs[sg.narrow] + sg.narrow_off;
        gm = unsigned(reinterpret_cast<uintptr_t>(si[k].src) & 15u);
        a |= unsigned(reinterpret_cast<uintptr_t>(si[k].src));
      } else {
        si[k].off = sg.narrow_off;
        const uint32_t g0 = p.goff[sg.narrow];
        if (!same) si[k].rcnt = p.goff[sg.narrow + 1] - g0;
        gm = unsigned(reinterpret_cast<uintptr_t>(p.bufs[p.gbuf[g0]] + sg.narrow_off) & 15u);
        a |= gm;
      }
      if (same) {
        // a segment whose narrow start moved mod 16 has its granules replanned
        si[k].moved = si[k].moved | (gm != si[k].gmis ? 1u : 0u);
      } else {
        si[k].nbytes = sg.width * nr;
        si[k].col = sg.col;
        si[k].units = sg.width;  // bytes for now
        si[k].moved = 0;
      }
      si[k].gmis = gm;
      atomicOr(&s_align, a);
    }
    if (!follows) __syncthreads();  // uniform
    if (DB && !gather) {
      // this block's image (every thread polls; the outcome is made uniform)
      const bool landed = staging::mbar_wait(&s_bar[buf], (parity >> buf) & 1u,
                                             staging::kWaitPolls);
      parity ^= 1u << buf;
      pending &= ~(1u << buf);
      ++nscatter;
      if (!__syncthreads_and(landed)) {
        // give the other image's load, if one is on its way, its own bounded wait
        if ((pending >> (buf ^ 1u)) & 1u)
          staging::mbar_wait(&s_bar[buf ^ 1u], (parity >> (buf ^ 1u)) & 1u, staging::kWaitPolls);
        if (threadIdx.x == 0) {
          atomicExch(p.status, staging::kStatusConsumerWait);
          staging::bulk_wait_all();
        }
        return;
      }
    }
    if (!follows && (s_align & uint32_t(U - 1)) != 0) {
      if (threadIdx.x == 0) atomicExch(p.status, staging::kStatusTransposeAlign);
      have_plan = false;
      continue;  // uniform: every thread read the same s_align
    }
    const bool replan = !same;
    if (replan) {
      if (threadIdx.x < 32) {
        // granules and replica pointer slots, exclusive prefix in segment order:
        // each lane owns segments [4 lane, 4 lane + 4) (K <= 128), then a warp scan.
        // A segment gets as many granules as its narrow range can touch at any
        // start mod 16, so the numbering holds for every block of the same shape
        // (the granules a start does not touch are empty).
        const int lane = int(threadIdx.x);
        uint32_t rc[4], gc[4], rsum = 0, gsum = 0;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t k = uint32_t(4 * lane + q);
          rc[q] = (k < K && !gather) ? si[k].rcnt : 0u;
          gc[q] = k < K ? (si[k].nbytes + 30u) >> 4 : 0u;
          rsum += rc[q];
          gsum += gc[q];
        }
        uint32_t rinc = rsum, ginc = gsum;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
          const uint32_t b = __shfl_up_sync(0xffffffffu, rinc, d);
          const uint32_t c = __shfl_up_sync(0xffffffffu, ginc, d);
          if (lane >= d) {
            rinc += b;
            ginc += c;
          }
        }
        uint32_t rb = rinc - rsum, gs = ginc - gsum;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t k = uint32_t(4 * lane + q);
          if (k < K) {
            if (!same) si[k].units /= U;
            si[k].rbeg = rb;
            si[k].gstart = gs;
            si[k].moved = 0;
          }
          rb += rc[q];
          gs += gc[q];
        }
        if (lane == 31) s_ngran = ginc;
      }
      __syncthreads();
      for (uint32_t k = threadIdx.x; k < K; k += kTThreads) {
        if (!same) fastdiv_init(si[k].units, &si[k].m, &si[k].l);
        if (!gather) {
          const uint32_t g0 = p.goff[p.segs[blk.seg_begin + k].narrow];
          for (uint32_t r = 0; r < si[k].rcnt; ++r) ptrs[si[k].rbeg + r] = p.bufs[p.gbuf[g0 + r]];
        }
      }
      __syncthreads();
    }
    const uint32_t ngran = s_ngran;
    // this thread's plans: made for a new shape, redone for segments that moved
#pragma unroll
    for (int sl = 0; sl < kSlots; ++sl) {
      const uint32_t g = threadIdx.x + uint32_t(sl) * kTThreads;
      if (g >= ngran) {
        plan[sl] = 0u;  // kind none
      } else if (replan) {
        const uint32_t k = uint32_t(find_granule(si, int(K), g));
        plan[sl] = plan_of<U>(si[k], k, g - si[k].gstart, L);
      } else {
        const uint32_t k = plan_k(plan[sl]);
        if (si[k].moved) plan[sl] = plan_of<U>(si[k], k, g - si[k].gstart, L);
      }
    }
    have_plan = true;
    // granules beyond the planned slots (blocks of unusually many granules)
    const uint32_t g_extra = uint32_t(kSlots) * kTThreads;

    if (gather) {
      // each thread loads whole aligned 16-byte granules of the segments' dense
      // source ranges (all its slots in flight) and puts their elements into the
      // image columns they belong to
      uint32_t unused[4] = {0u, 0u, 0u, 0u};
      constexpr int kHalf = kSlots / 2;
#pragma unroll
      for (int h0 = 0; h0 < kSlots; h0 += kHalf) {
        uint4 v[kHalf];
#pragma unroll
        for (int q = 0; q < kHalf; ++q) {
          const uint32_t meta = plan[h0 + q];
          if (plan_kind(meta) != kKindNone) {
            const SegInfo& s = si[plan_k(meta)];
            const uint32_t g = threadIdx.x + uint32_t(h0 + q) * kTThreads;
            v[q] = narrow_load(s.src - s.gmis + 16 * size_t(g - s.gstart));
          }
        }
        if (h0 == 0) {
          // this thread's partial granule (threads < 2 K), while its loads are in flight
          uint32_t k, j;
          if (threadIdx.x < 2 * K && edge_granule<U>(si, threadIdx.x, &k, &j)) {
            const SegInfo& s = si[k];
            const uint32_t meta = plan_of<U, true>(s, k, j, L);
            if (plan_kind(meta) != kKindNone) {
              uint32_t lo, hi;
              granule_span(s, j, &lo, &hi);
              const uint4 w = narrow_load(s.src - s.gmis + 16 * size_t(j));
              granule_move<U, true>(s, meta, lo, hi, img + mis + plan_off(meta), L, unused, w);
            }
          }
        }
#pragma unroll
        for (int q = 0; q < kHalf; ++q) {
          const uint32_t meta = plan[h0 + q];
          if (plan_kind(meta) == kKindNone) continue;
          const SegInfo& s = si[plan_k(meta)];
          uint32_t lo = 0u, hi = 16u;
          if (plan_kind(meta) == kKindWalk) {
            const uint32_t g = threadIdx.x + uint32_t(h0 + q) * kTThreads;
            granule_span(s, g - s.gstart, &lo, &hi);
          }
          granule_move<U, true>(s, meta, lo, hi, img + mis + plan_off(meta), L, unused, v[q]);
        }
      }
      // whole granules beyond the planned slots, then the partial ones
      for (uint32_t g = g_extra + threadIdx.x; g < ngran; g += kTThreads) {
        const uint32_t k = uint32_t(find_granule(si, int(K), g));
        const SegInfo& s = si[k];
        const uint32_t meta = plan_of<U>(s, k, g - s.gstart, L);
        if (plan_kind(meta) == kKindNone) continue;
        uint32_t lo, hi;
        granule_span(s, g - s.gstart, &lo, &hi);
        const uint4 w = narrow_load(s.src - s.gmis + 16 * size_t(g - s.gstart));
        granule_move<U, true>(s, meta, lo, hi, img + mis + plan_off(meta), L, unused, w);
      }
      // the image's bytes become visible to the bulk copies' (async) proxy
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncthreads();
      // image [mis, mis + n) -> each replica's [wide_off, wide_off + n): the aligned
      // middle by one bulk copy per replica (thread 0; the image is not written
      // again before thread 0 has seen the copies read it), the partial head and
      // tail granules by the threads
      const uint32_t h = min((16u - mis) & 15u, n);
      const uint32_t m16 = (n - h) >> 4;
      for (int r = 0; r < R; ++r) {
        unsigned char* d = ptrs[r] + blk.wide_off;
        const bool vec = congruent || ((reinterpret_cast<uintptr_t>(d) & 15u) == mis);
        if (!vec) {
          for (uint32_t i = threadIdx.x; i < n; i += kTThreads) d[i] = img[mis + i];
          continue;
        }
        for (uint32_t i = threadIdx.x; i < h; i += kTThreads) d[i] = img[mis + i];
        if (m16 != 0 && threadIdx.x == 0) bulk_store_evict_first(d + h, img + mis + h, 16u * m16);
        for (uint32_t i = h + 16 * m16 + threadIdx.x; i < n; i += kTThreads) d[i] = img[mis + i];
      }
      if (threadIdx.x == 0) staging::bulk_commit();
    } else {
      if constexpr (!DB) {
        // wide rows -> image, 16-byte loads from the aligned granules holding them
        const unsigned char* base = wsrc - mis;
        const uint32_t nv = (mis + n + 15u) >> 4;
#pragma unroll 1
        for (uint32_t k0 = threadIdx.x; k0 < nv; k0 += kTThreads * kTVecUnroll) {
          uint4 v[kTVecUnroll];
#pragma unroll
          for (int j = 0; j < kTVecUnroll; ++j) {
            const uint32_t k = k0 + j * kTThreads;
            if (k < nv) v[j] = __ldcs(reinterpret_cast<const uint4*>(base + 16 * k));
          }
#pragma unroll
          for (int j = 0; j < kTVecUnroll; ++j) {
            const uint32_t k = k0 + j * kTThreads;
            if (k < nv) *reinterpret_cast<uint4*>(img + 16 * k) = v[j];
          }
        }
        __syncthreads();
      }
      // (DB: the wide rows arrived by the bulk copy waited for above)
      // each thread builds whole 16-byte granules of the segments' dense destination
      // ranges (aligned like replica 0) from the image and writes them to every
      // replica of the segment
      const uint4 none = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll 1
      for (int sl = 0; sl < kSlots; ++sl) {
        // The loop is rolled: its body, with every granule kind inlined, exists once
        // instead of once per slot (unrolled, the warps stalled on instruction
        // fetch; the gather's loop stays unrolled, its loads of several slots in
        // flight together).  This slot's plan is plan[0]: rotating the plans left
        // each slot (kSlots rotations restore their order for the next block) keeps
        // them in registers at one move each.
        const uint32_t meta = plan[0];
#pragma unroll
        for (int q = 0; q + 1 < kSlots; ++q) plan[q] = plan[q + 1];
        plan[kSlots - 1] = meta;
        if (sl == 1) {
          // this thread's partial granule (threads < 2 K), between its planned ones so
          // that it overlaps the other warps' work
          uint32_t k, j;
          if (threadIdx.x < 2 * K && edge_granule<U>(si, threadIdx.x, &k, &j)) {
            const SegInfo& s = si[k];
            const uint32_t meta = plan_of<U, true>(s, k, j, L);
            if (plan_kind(meta) != kKindNone) {
              uint32_t lo, hi;
              granule_span(s, j, &lo, &hi);
              uint32_t words[4] = {0u, 0u, 0u, 0u};
              granule_move<U, false>(s, meta, lo, hi, img + mis + plan_off(meta), L, words, none);
              scatter_store(s, j, lo, hi, words, ptrs);
            }
          }
        }
        if (plan_kind(meta) == kKindNone) continue;
        const SegInfo& s = si[plan_k(meta)];
        const uint32_t j = threadIdx.x + uint32_t(sl) * kTThreads - s.gstart;
        uint32_t words[4] = {0u, 0u, 0u, 0u};
        if (plan_kind(meta) != kKindWalk) {
          // a whole granule: with one replica, one aligned store
          granule_move<U, false>(s, meta, 0u, 16u, img + mis + plan_off(meta), L, words, none);
          if (s.rcnt == 1)
            __stcs(reinterpret_cast<uint4*>(ptrs[s.rbeg] + s.off - s.gmis + 16 * size_t(j)),
                   make_uint4(words[0], words[1], words[2], words[3]));
          else
            scatter_store(s, j, 0u, 16u, words, ptrs);
        } else {
          uint32_t lo, hi;
          granule_span(s, j, &lo, &hi);
          granule_move<U, false>(s, meta, lo, hi, img + mis + plan_off(meta), L, words, none);
          scatter_store(s, j, lo, hi, words, ptrs);
        }
      }
      // whole granules beyond the planned slots, then the partial ones
      for (uint32_t g = g_extra + threadIdx.x; g < ngran; g += kTThreads) {
        const uint32_t k = uint32_t(find_granule(si, int(K), g));
        const SegInfo& s = si[k];
        const uint32_t meta = plan_of<U>(s, k, g - s.gstart, L);
        if (plan_kind(meta) == kKindNone) continue;
        uint32_t lo, hi;
        granule_span(s, g - s.gstart, &lo, &hi);
        uint32_t words[4] = {0u, 0u, 0u, 0u};
        granule_move<U, false>(s, meta, lo, hi, img + mis + plan_off(meta), L, words, none);
        scatter_store(s, g - s.gstart, lo, hi, words, ptrs);
      }
    }
  }
  if (threadIdx.x == 0) staging::bulk_wait_all();  // the last gather block's bulk stores
}

std::mutex g_t_mu;
std::map<std::pair<int, int>, int> g_t_occ;  // (device, 2 log2 U + DB) -> blocks per SM

using TransposeFn = void (*)(TransposeParams);
const TransposeFn kTransposeKernels[2][4] = {
    {reshard_transpose_kernel<1, false>, reshard_transpose_kernel<2, false>,
     reshard_transpose_kernel<4, false>, reshard_transpose_kernel<8, false>},
    {reshard_transpose_kernel<1, true>, reshard_transpose_kernel<2, true>,
     reshard_transpose_kernel<4, true>, reshard_transpose_kernel<8, true>}};

}  // namespace

reshard_status_t launch_transposes(const reshard_plan_s* plan, const Program& prog,
                                   unsigned char* const* bufs, int nbufs, uint32_t flags,
                                   void* stream) {
  if (prog.tblocks.empty()) return RESHARD_OK;
  int dev = -1;
  cudaError_t ce = cudaGetDevice(&dev);
  if (ce != cudaSuccess)
    return fail(RESHARD_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(ce));
  // element width: the widest of 1, 2, 4, 8 bytes that divides every row length,
  // column, width and offset of the blocks and every buffer's address
  uint64_t bits = prog.talign_bits | 8u;
  for (int i = 0; i < nbufs; ++i) bits |= uint64_t(reinterpret_cast<uintptr_t>(bufs[i]));
  const int ulog = (bits & 1u) ? 0 : (bits & 2u) ? 1 : (bits & 4u) ? 2 : 3;
  const int db = prog.tscatter ? 1 : 0;
  const int smem = db ? dyn_smem<true>() : dyn_smem<false>();
  const void* fn = reinterpret_cast<const void*>(kTransposeKernels[db][ulog]);
  int bps = 0;
  {
    std::lock_guard<std::mutex> lk(g_t_mu);
    auto it = g_t_occ.find({dev, 2 * ulog + db});
    if (it == g_t_occ.end()) {
      ce = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (ce == cudaSuccess)
        ce = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bps, fn, kTThreads, smem);
      if (ce != cudaSuccess)
        return fail(RESHARD_ERR_CUDA, std::string("transpose kernel set-up: ") + cudaGetErrorString(ce));
      bps = bps > 0 ? bps : 1;
      g_t_occ[{dev, 2 * ulog + db}] = bps;
    } else {
      bps = it->second;
    }
  }
  unsigned int* status = nullptr;
  reshard_status_t st = device_status_word(&status);
  if (st != RESHARD_OK) return st;
  TransposeParams tp;
  tp.status = status;
  tp.blocks = prog.d_tblocks;
  tp.segs = prog.d_tsegs;
  tp.goff = prog.d_goff;
  tp.gbuf = prog.d_gbuf;
  tp.nblocks = int64_t(prog.tblocks.size());
  tp.nbufs = nbufs;
  tp.flags = flags;
  for (int i = 0; i < nbufs; ++i) tp.bufs[i] = bufs[i];
  for (int i = nbufs; i < RESHARD_MAX_EXEC_BUFFERS; ++i) tp.bufs[i] = nullptr;
  const int64_t max_grid = int64_t(plan->num_sms) * bps;
  const unsigned grid = unsigned(tp.nblocks < max_grid ? tp.nblocks : max_grid);
  void* args[] = {&tp};
  ce = cudaLaunchKernel(fn, dim3(grid), dim3(kTThreads), args, size_t(smem),
                        static_cast<cudaStream_t>(stream));
  if (ce != cudaSuccess)
    return fail(RESHARD_ERR_CUDA, std::string("kernel launch: ") + cudaGetErrorString(ce));
  return RESHARD_OK;
}

}  // namespace rs
