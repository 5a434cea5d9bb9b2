// kernels.cu -- the vector copy kernel of libreshard.so (sm_103a).
//
// One persistent kernel executes every copy program of a plan: the read-once
// fan-out reshard, the per-replica box copy, and both steps of the
// gather-and-broadcast baseline.  (A fan-out whose tiles and buffers are all
// 16-byte aligned is handed to the TMA-staged kernel of bulk_fanout.cu, which
// uses the same work partition.)  The work of a program is a list of tiles
// (see reshard_tile_t), each split into equal work units; CTA b of a grid of
// G takes units [b*U/G, (b+1)*U/G) of the program's U units, so every CTA
// moves the same number of bytes regardless of how unequal the tiles are, and
// consecutive CTAs walk consecutive destination addresses.
//
// Within a tile a CTA streams 16-byte vectors (narrower when the runtime
// addresses, strides or row length are not 16-byte aligned): every thread
// issues several independent loads before it stores (about 64 bytes in flight
// per thread whatever the vector width), and each loaded vector is
// stored to every destination buffer of the tile's group (the fan-out: the
// source region is read from HBM once, written R times).  Loads and stores use
// the normal cache policy (see load_stream).
//
// There is no tensor-core work here: a reshard is a pure byte copy, bounded by
// HBM bandwidth.
#include <cuda_runtime.h>

#include <cstdint>
#include <map>
#include <mutex>
#include <string>
#include <utility>

#include "internal.h"
#include "staging.cuh"

namespace rs {
namespace {

constexpr int kThreads = 256;
// Independent loads each thread keeps in flight: about kInflightBytes per
// thread whatever the access width (at most 16 loads), so that narrow accesses
// still keep enough bytes in flight to cover the memory latency.
constexpr int kInflightBytes = 64;
template <int W> __host__ __device__ constexpr int unroll_of() {
  return kInflightBytes / W < 4 ? 4 : (kInflightBytes / W > 16 ? 16 : kInflightBytes / W);
}

// Unsigned 32-bit division by a runtime-invariant divisor through a multiply
// and a shift (Granlund and Montgomery, "Division by Invariant Integers using
// Multiplication", PLDI 1994, round-up method): for d >= 1 with
// l = ceil(log2 d) and m = floor(2^32 (2^l - d) / d) + 1,
// n / d = (umulhi(n, m) + n) >> l for every 32-bit n.
struct FastDiv {
  uint32_t d, m, l;
  __device__ __forceinline__ explicit FastDiv(uint32_t div) : d(div) {
    l = 0;
    while ((uint64_t(1) << l) < div) ++l;
    m = uint32_t(((uint64_t(1) << 32) * ((uint64_t(1) << l) - div)) / div + 1);
  }
  __device__ __forceinline__ uint32_t div(uint32_t n) const {
    return uint32_t((uint64_t(__umulhi(n, m)) + n) >> l);
  }
};

template <int W> struct Vec;
template <> struct Vec<16> { using T = uint4; };
template <> struct Vec<8> { using T = uint2; };
template <> struct Vec<4> { using T = unsigned int; };
template <> struct Vec<2> { using T = unsigned short; };
template <> struct Vec<1> { using T = unsigned char; };

// Loads and stores of the element kernel keep the normal cache policy: rows that
// do not start or end on a 32-byte sector share those sectors with other tiles,
// which evict-first accesses dropped from L2 before the other tile's access
// (measured per tensor: 12-20% on short-row scatters and gathers, no change on
// long runs).
template <typename T>
__device__ __forceinline__ T load_stream(const unsigned char* p) {
  return *reinterpret_cast<const T*>(p);
}
template <typename T>
__device__ __forceinline__ void store_stream(unsigned char* p, const T& v) {
  *reinterpret_cast<T*>(p) = v;
}
// The register realigning kernel's stores stay evict-first (measured 3% faster
// there on a 6-replica fan-out of 13 KB rows).
__device__ __forceinline__ void store_evict_first(unsigned char* p, const uint4& v) {
  __stcs(reinterpret_cast<uint4*>(p), v);
}

// Bytes [0, nbytes) of a contiguous run: from src to dst + dofs for each of
// the R destination buffers dst in sdst.
template <int W, int kUnroll>
__device__ __forceinline__ void copy_run(const unsigned char* __restrict__ src,
                                         unsigned char* const* sdst, int R, int64_t dofs,
                                         uint32_t nbytes) {
  using V = typename Vec<W>::T;
  const uint32_t n = nbytes / W;
#pragma unroll 1
  for (uint32_t base = threadIdx.x; base < n; base += kThreads * kUnroll) {
    V v[kUnroll];
#pragma unroll
    for (int k = 0; k < kUnroll; ++k) {
      const uint32_t i = base + k * kThreads;
      if (i < n) v[k] = load_stream<V>(src + size_t(i) * W);
    }
#pragma unroll 1
    for (int r = 0; r < R; ++r) {
      unsigned char* d = sdst[r] + dofs;
#pragma unroll
      for (int k = 0; k < kUnroll; ++k) {
        const uint32_t i = base + k * kThreads;
        if (i < n) store_stream<V>(d + size_t(i) * W, v[k]);
      }
    }
  }
}

// Rows [r_begin, r_end) of a multi-row tile.  The row index runs over
// planes x rows: row r = p * nrows + q starts at src + p*sps + q*srs and at
// dofs + p*dps + q*drs in every destination (PLANES = false: one plane).
// Rows are vpr vectors of W bytes.  Rows of at least kThreads vectors are
// streamed as one flat range of vectors by the whole CTA; shorter rows are packed
// kThreads / vpr to a pass, one thread per vector, and every thread carries
// kUnroll rows at once.
template <int W, bool PLANES, int kUnroll>
__device__ __forceinline__ void copy_rows(const reshard_tile_t& t, const unsigned char* src,
                                          unsigned char* const* sdst, int R, uint32_t r_begin,
                                          uint32_t r_end) {
  using V = typename Vec<W>::T;
  const uint32_t vpr = t.row_bytes / W;
  const FastDiv by_rows(PLANES ? t.nrows : 1u);
  const unsigned char* s0 = src + t.src_off;
  auto src_row = [&](uint32_t r) -> int64_t {
    if (!PLANES) return int64_t(r) * t.src_row_stride;
    const uint32_t p = by_rows.div(r);
    return int64_t(p) * t.src_plane_stride + int64_t(r - p * t.nrows) * t.src_row_stride;
  };
  auto dst_row = [&](uint32_t r) -> int64_t {
    if (!PLANES) return int64_t(r) * t.dst_row_stride;
    const uint32_t p = by_rows.div(r);
    return int64_t(p) * t.dst_plane_stride + int64_t(r - p * t.nrows) * t.dst_row_stride;
  };
  if (vpr >= uint32_t(kThreads)) {
    // long rows: the block walks (row, vector) pairs flat, kThreads vectors apart,
    // so every thread keeps its loads in flight whatever the row length.  As
    // vpr >= kThreads a step crosses at most one row boundary.  The store cursor
    // repeats the load cursor's walk instead of holding one offset per load.
    uint32_t lrow = r_begin, lcol = threadIdx.x;
    int64_t lbase = src_row(lrow);
    uint32_t srow = r_begin, scol = threadIdx.x;
    int64_t sbase = t.dst_off + dst_row(srow);
#pragma unroll 1
    while (lrow < r_end) {
      V v[kUnroll];
#pragma unroll
      for (int k = 0; k < kUnroll; ++k) {
        if (lrow < r_end) v[k] = load_stream<V>(s0 + lbase + int64_t(lcol) * W);
        lcol += kThreads;
        if (lcol >= vpr) {
          lcol -= vpr;
          lbase = src_row(++lrow);
        }
      }
#pragma unroll
      for (int k = 0; k < kUnroll; ++k) {
        if (srow < r_end) {
          const int64_t d = sbase + int64_t(scol) * W;
#pragma unroll 1
          for (int j = 0; j < R; ++j) store_stream<V>(sdst[j] + d, v[k]);
        }
        scol += kThreads;
        if (scol >= vpr) {
          scol -= vpr;
          sbase = t.dst_off + dst_row(++srow);
        }
      }
    }
    return;
  }
  const uint32_t step = uint32_t(kThreads) / vpr;  // rows per pass
  const uint32_t rsub = threadIdx.x / vpr;
  const uint32_t c = threadIdx.x - rsub * vpr;
  if (rsub >= step) return;  // the last threads idle when vpr does not divide kThreads
  const unsigned char* s = s0 + int64_t(c) * W;
  const int64_t d0 = t.dst_off + int64_t(c) * W;
#pragma unroll 1
  for (uint32_t row = r_begin + rsub; row < r_end; row += step * kUnroll) {
    V v[kUnroll];
#pragma unroll
    for (int k = 0; k < kUnroll; ++k) {
      const uint32_t r = row + k * step;
      if (r < r_end) v[k] = load_stream<V>(s + src_row(r));
    }
#pragma unroll 1
    for (int j = 0; j < R; ++j) {
      unsigned char* d = sdst[j] + d0;
#pragma unroll
      for (int k = 0; k < kUnroll; ++k) {
        const uint32_t r = row + k * step;
        if (r < r_end) store_stream<V>(d + dst_row(r), v[k]);
      }
    }
  }
}

// NARROW: programs whose bytes are mostly in rows under kNarrowRow bytes keep 4
// loads in flight per thread: each load there already pulls a whole sector of
// the source, and more of them in flight were measured slower (4-byte rows at
// a 32-byte source stride: 0.15 -> 0.21 ms with 16).
template <int W, bool PLANES, bool NARROW>
__global__ void __launch_bounds__(kThreads, PLANES ? 2 : 4)
    reshard_copy_kernel(const __grid_constant__ KernelParams p) {
  constexpr int kUnroll = NARROW ? 4 : unroll_of<W>();
  __shared__ unsigned char* s_dst[kMaxGroup];

  const int64_t total = p.total_units;
  int64_t u0 = total * int64_t(blockIdx.x) / int64_t(gridDim.x);
  const int64_t u1 = total * int64_t(blockIdx.x + 1) / int64_t(gridDim.x);
  if (u0 >= u1) return;

  // largest tile index t with prefix[t] <= u0
  int lo = 0, hi = p.ntiles - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.prefix[mid] <= u0) lo = mid;
    else hi = mid - 1;
  }
  int ti = lo;

  while (u0 < u1) {
    const reshard_tile_t t = p.tiles[ti];
    const int64_t tb = p.prefix[ti];
    const int64_t te = p.prefix[ti + 1];
    const int64_t a = u0 - tb;
    const int64_t b = (u1 < te ? u1 : te) - tb;

    const uint32_t g0 = p.goff[t.dst_group];
    const int R = int(p.goff[t.dst_group + 1] - g0);
    __syncthreads();  // previous tile's readers of s_dst are done
    for (int i = threadIdx.x; i < R; i += kThreads) s_dst[i] = p.bufs[p.gbuf[g0 + i]];
    __syncthreads();

    const unsigned char* src = p.bufs[t.src_buf];
    if (t.nrows == 1 && t.nplanes == 1) {
      const int64_t b0 = a * kUnitBytes;
      const int64_t b1 = min(b * kUnitBytes, int64_t(t.row_bytes));
      copy_run<W, kUnroll>(src + t.src_off + b0, s_dst, R, t.dst_off + b0, uint32_t(b1 - b0));
    } else {
      const uint32_t upr = rows_per_unit(t.row_bytes);
      const uint64_t rows = uint64_t(t.nrows) * t.nplanes;
      const uint32_t r_begin = uint32_t(a * upr);
      const uint32_t r_end = uint32_t(min(uint64_t(b) * upr, rows));
      if (PLANES && t.nplanes > 1) copy_rows<W, true, kUnroll>(t, src, s_dst, R, r_begin, r_end);
      else copy_rows<W, false, kUnroll>(t, src, s_dst, R, r_begin, r_end);
    }
    u0 = tb + b;
    ++ti;
  }
}


// ---------------------------------------------------------------- realigning path
// For programs whose offsets, strides or rows are not all 16-byte aligned.  A
// destination range is written with aligned 16-byte stores; each output
// vector is assembled from the two aligned 16-byte source vectors that hold
// its bytes (byte permute), so source and destination may differ in alignment
// by any number of bytes.  Bytes before the first and after the last aligned
// destination vector are copied one by one.  Source reads may touch bytes
// outside the range only inside the aligned 16-byte granules that also hold
// bytes of the range.

__device__ __forceinline__ uint4 load16_cached(const unsigned char* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}

using staging::funnel16;

constexpr int kRealignUnroll = 4;

// m aligned destination vectors: vector k comes from source bytes at base + o + 16k.
__device__ __forceinline__ void realigned_body(const unsigned char* base, uint32_t o,
                                               unsigned char* const* sdst, int R, int64_t doff,
                                               uint32_t m, int tid, int nthr) {
  const uint32_t q = o >> 2;
  const uint32_t sel = 0x3210u + 0x1111u * (o & 3u);
  const bool two = o != 0;
#pragma unroll 1
  for (uint32_t k0 = tid; k0 < m; k0 += uint32_t(kRealignUnroll) * nthr) {
    uint4 out[kRealignUnroll];
#pragma unroll
    for (int j = 0; j < kRealignUnroll; ++j) {
      const uint32_t k = k0 + j * nthr;
      if (k < m) {
        const uint4 A = load16_cached(base + size_t(k) * 16);
        const uint4 B = two ? load16_cached(base + size_t(k) * 16 + 16) : A;
        out[j] = funnel16(A, B, q, sel);
      }
    }
#pragma unroll 1
    for (int r = 0; r < R; ++r) {
      unsigned char* d = sdst[r] + doff;
#pragma unroll
      for (int j = 0; j < kRealignUnroll; ++j) {
        const uint32_t k = k0 + j * nthr;
        if (k < m) store_evict_first(d + size_t(k) * 16, out[j]);
      }
    }
  }
}

// n bytes from s to sdst[r] + doff for r < R, by threads tid of nthr.  All
// sdst[r] + doff must have the same address mod 16.
__device__ __forceinline__ void realigned_copy(const unsigned char* s, unsigned char* const* sdst,
                                               int R, int64_t doff, uint64_t n, int tid,
                                               int nthr) {
  const uint32_t dmis = uint32_t(reinterpret_cast<uintptr_t>(sdst[0] + doff) & 15u);
  const uint64_t h = min(uint64_t((16u - dmis) & 15u), n);
  for (uint64_t i = tid; i < h; i += nthr) {
    const unsigned char v = s[i];
    for (int r = 0; r < R; ++r) sdst[r][doff + i] = v;
  }
  const uint32_t m = uint32_t((n - h) >> 4);
  const unsigned char* s0 = s + h;
  const uint32_t o = uint32_t(reinterpret_cast<uintptr_t>(s0) & 15u);
  const unsigned char* base = s0 - o;
  realigned_body(base, o, sdst, R, doff + int64_t(h), m, tid, nthr);
  for (uint64_t i = h + uint64_t(m) * 16 + tid; i < n; i += nthr) {
    const unsigned char v = s[i];
    for (int r = 0; r < R; ++r) sdst[r][doff + i] = v;
  }
}

// A short row (< 64 bytes) by one thread, in the widest unit both ends allow.
__device__ __forceinline__ void short_row_copy(const unsigned char* s, unsigned char* d,
                                               uint32_t n) {
  const uint32_t a = uint32_t(reinterpret_cast<uintptr_t>(s) | reinterpret_cast<uintptr_t>(d)) | n;
  if ((a & 7u) == 0) {
    for (uint32_t i = 0; i < n; i += 8)
      *reinterpret_cast<uint2*>(d + i) = *reinterpret_cast<const uint2*>(s + i);
  } else if ((a & 3u) == 0) {
    for (uint32_t i = 0; i < n; i += 4)
      *reinterpret_cast<uint32_t*>(d + i) = *reinterpret_cast<const uint32_t*>(s + i);
  } else if ((a & 1u) == 0) {
    for (uint32_t i = 0; i < n; i += 2)
      *reinterpret_cast<uint16_t*>(d + i) = *reinterpret_cast<const uint16_t*>(s + i);
  } else {
    for (uint32_t i = 0; i < n; ++i) d[i] = s[i];
  }
}

constexpr uint32_t kShortRow = 64;

template <bool PLANES>
__global__ void __launch_bounds__(kThreads, PLANES ? 2 : 3)
    reshard_realign_kernel(const __grid_constant__ KernelParams p) {
  __shared__ unsigned char* s_dst[kMaxGroup];
  const bool congruent = (p.flags & kFlagDstCongruent) != 0;
  const int64_t total = p.total_units;
  int64_t u0 = total * int64_t(blockIdx.x) / int64_t(gridDim.x);
  const int64_t u1 = total * int64_t(blockIdx.x + 1) / int64_t(gridDim.x);
  if (u0 >= u1) return;
  int lo = 0, hi = p.ntiles - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.prefix[mid] <= u0) lo = mid;
    else hi = mid - 1;
  }
  int ti = lo;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  while (u0 < u1) {
    const reshard_tile_t t = p.tiles[ti];
    const int64_t tb = p.prefix[ti];
    const int64_t te = p.prefix[ti + 1];
    const int64_t a = u0 - tb;
    const int64_t b = (u1 < te ? u1 : te) - tb;
    const uint32_t g0 = p.goff[t.dst_group];
    const int R = int(p.goff[t.dst_group + 1] - g0);
    __syncthreads();
    for (int i = threadIdx.x; i < R; i += kThreads) s_dst[i] = p.bufs[p.gbuf[g0 + i]];
    __syncthreads();
    const unsigned char* src = p.bufs[t.src_buf];
    const bool run = t.nrows == 1 && t.nplanes == 1;
    const uint32_t upr = rows_per_unit(t.row_bytes);
    const uint64_t rows = uint64_t(t.nrows) * t.nplanes;
    const uint32_t r_begin = run ? 0u : uint32_t(a * upr);
    const uint32_t r_end = run ? 1u : uint32_t(min(uint64_t(b) * upr, rows));
    const FastDiv by_rows(PLANES ? t.nrows : 1u);
    auto row_offsets = [&](uint32_t r, int64_t* so, int64_t* dof) {
      uint32_t pl = 0, q = r;
      if (PLANES) {
        pl = by_rows.div(r);
        q = r - pl * t.nrows;
      }
      *so = t.src_off + int64_t(pl) * t.src_plane_stride + int64_t(q) * t.src_row_stride;
      *dof = t.dst_off + int64_t(pl) * t.dst_plane_stride + int64_t(q) * t.dst_row_stride;
    };
    if (run || t.row_bytes >= kShortRow) {
      // a run: the whole CTA on its byte range; long rows: one warp per row
      const uint32_t njobs = r_end - r_begin;
      const uint32_t first = run ? 0u : uint32_t(warp);
      const uint32_t stride = run ? 1u : uint32_t(kThreads / 32);
      const int tid = run ? int(threadIdx.x) : lane;
      const int nthr = run ? kThreads : 32;
      for (uint32_t j = first; j < njobs; j += stride) {
        int64_t so, dof;
        uint64_t n;
        if (run) {
          const int64_t b0 = a * kUnitBytes;
          so = t.src_off + b0;
          dof = t.dst_off + b0;
          n = uint64_t(min(b * kUnitBytes, int64_t(t.row_bytes)) - b0);
        } else {
          row_offsets(r_begin + j, &so, &dof);
          n = t.row_bytes;
        }
        const int passes = congruent ? 1 : R;
        for (int q = 0; q < passes; ++q)
          realigned_copy(src + so, s_dst + q, congruent ? R : 1, dof, n, tid, nthr);
      }
    } else {
      // short rows: one thread per row
      for (uint32_t r = r_begin + threadIdx.x; r < r_end; r += kThreads) {
        int64_t so, dof;
        row_offsets(r, &so, &dof);
        for (int j = 0; j < R; ++j) short_row_copy(src + so, s_dst[j] + dof, t.row_bytes);
      }
    }
    u0 = tb + b;
    ++ti;
  }
}

using KernelFn = void (*)(KernelParams);

// choose_kernel's answer for the TMA-staged realigning kernel (realign_staged.cu).
constexpr int kStagedRealign = -1;
// Source bytes from which a fan-out program goes through that kernel, and
// from which a one-replica program with 4-byte elements does.
constexpr int64_t kStagedFanoutMinBytes = int64_t(48) << 20;
constexpr int64_t kStagedW4MinBytes = int64_t(128) << 20;
// Fan-out from which that kernel writes through bulk copies from an output
// stage (when most bytes are in rows of at least 8 KiB: a bulk copy per row
// and replica costs the copy engine about as much as 1 KB of streaming).
constexpr int kBulkStoreFanout = 2;

bool bulk_stores(const Program& prog) {
  return prog.max_fanout >= kBulkStoreFanout && 2 * prog.wide_row_bytes >= prog.tile_bytes;
}

// Instantiations indexed by [narrow rows][log2 W][planes].
// [0]: realigning kernel (any alignment); [k], k = 1..4: 2^k-byte vector kernel;
// [5]: byte kernel.
const KernelFn kKernels[2][6][2] = {
    {{reshard_realign_kernel<false>, reshard_realign_kernel<true>},
     {reshard_copy_kernel<2, false, false>, reshard_copy_kernel<2, true, false>},
     {reshard_copy_kernel<4, false, false>, reshard_copy_kernel<4, true, false>},
     {reshard_copy_kernel<8, false, false>, reshard_copy_kernel<8, true, false>},
     {reshard_copy_kernel<16, false, false>, reshard_copy_kernel<16, true, false>},
     {reshard_copy_kernel<1, false, false>, reshard_copy_kernel<1, true, false>}},
    {{reshard_realign_kernel<false>, reshard_realign_kernel<true>},
     {reshard_copy_kernel<2, false, true>, reshard_copy_kernel<2, true, true>},
     {reshard_copy_kernel<4, false, true>, reshard_copy_kernel<4, true, true>},
     {reshard_copy_kernel<8, false, true>, reshard_copy_kernel<8, true, true>},
     {reshard_copy_kernel<16, false, true>, reshard_copy_kernel<16, true, true>},
     {reshard_copy_kernel<1, false, true>, reshard_copy_kernel<1, true, true>}}};

// Kernel for a program whose widest common access is 2^w_log2 bytes (rule
// fitted to per-tensor timings of the uneven-stress tensors):
//   everything 16-byte aligned: the 16-byte vector kernel (or the TMA fan-out);
//   fan-out to several replicas: the TMA-staged realigning kernel with bulk
//     stores when most bytes are in rows of at least 8 KiB and the program is
//     large enough to fill its pipelines, else the register realigning kernel
//     when most bytes are in rows of at least 512 bytes;
//   one replica, rows of at least 512 bytes: the staged kernel when the
//     element width would be 1 or 2 bytes, or 4 bytes in a large program made
//     mostly of rows of at least 8 KiB (long runs: its loads stay wide whatever
//     the alignment; on 0.6-1.4 KB rows the element kernel, with 64 bytes in
//     flight per thread, was measured 11-29% faster);
//   otherwise the element-width kernel.
int choose_kernel(const Program& prog, int w_log2) {
  if (w_log2 == 4) return 4;
  const bool long_rows = 2 * prog.long_row_bytes >= prog.tile_bytes;
  const bool wide_rows = 2 * prog.wide_row_bytes >= prog.tile_bytes;
  if (prog.max_fanout >= 2) {
    if (wide_rows && prog.tile_bytes >= kStagedFanoutMinBytes) return kStagedRealign;
    if (long_rows) return 0;
  } else if (long_rows && (w_log2 <= 1 || (w_log2 == 2 && wide_rows &&
                                            prog.tile_bytes >= kStagedW4MinBytes))) {
    return kStagedRealign;
  }
  return w_log2 == 0 ? 5 : w_log2;
}

// Every destination buffer of the program at the same address mod 16?
bool destinations_congruent(const Program& prog, unsigned char* const* bufs) {
  int64_t first = -1;
  for (uint16_t bi : prog.gbuf) {
    const int64_t m = int64_t(reinterpret_cast<uintptr_t>(bufs[bi]) & 15u);
    if (bufs[bi] == nullptr) continue;
    if (first < 0) first = m;
    else if (m != first) return false;
  }
  return true;
}

std::mutex g_occ_mu;
std::map<std::pair<int, int>, int> g_occ;  // (device, kernel index) -> blocks per SM

reshard_status_t occupancy(int device, int w_log2, int planes, int narrow, int* blocks) {
  const std::pair<int, int> key(device, (narrow * 6 + w_log2) * 2 + planes);
  std::lock_guard<std::mutex> lk(g_occ_mu);
  auto it = g_occ.find(key);
  if (it != g_occ.end()) {
    *blocks = it->second;
    return RESHARD_OK;
  }
  int n = 0;
  cudaError_t ce = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
      &n, reinterpret_cast<const void*>(kKernels[narrow][w_log2][planes]), kThreads, 0);
  if (ce != cudaSuccess)
    return fail(RESHARD_ERR_CUDA, std::string("occupancy query: ") + cudaGetErrorString(ce));
  n = n > 0 ? n : 1;
  g_occ[key] = n;
  *blocks = n;
  return RESHARD_OK;
}

}  // namespace

Dispatch decide(const Program& prog, unsigned char* const* bufs, int nbufs, bool allow_tma_fanout) {
  Dispatch d;
  if (prog.total_units() == 0) return d;
  // widest access every tile of the program allows with these buffers
  uint64_t align = prog.align_bits;
  for (int i = 0; i < nbufs; ++i) align |= reinterpret_cast<uint64_t>(bufs[i]);
  d.w_log2 = 4;
  while (d.w_log2 > 0 && (align & ((uint64_t(1) << d.w_log2) - 1)) != 0) --d.w_log2;
  d.flags = destinations_congruent(prog, bufs) ? kFlagDstCongruent : 0u;
  if (allow_tma_fanout && prog.staged && d.w_log2 == 4) {
    d.path = RESHARD_PATH_TMA_FANOUT;
    return d;
  }
  d.kidx = choose_kernel(prog, d.w_log2);
  d.narrow = 2 * prog.narrow_row_bytes >= prog.tile_bytes ? 1 : 0;
  if (d.kidx == kStagedRealign) {
    if (bulk_stores(prog)) d.flags |= kFlagBulkStores;
    d.path = (d.flags & kFlagDstCongruent) && (d.flags & kFlagBulkStores)
                 ? RESHARD_PATH_STAGED_BULK
                 : RESHARD_PATH_STAGED;
  } else if (d.kidx == 0) {
    d.path = RESHARD_PATH_REALIGN;
  } else {
    d.path = RESHARD_PATH_VECTOR;
  }
  return d;
}

reshard_status_t copy_kernel_occupancy(int* blocks_per_sm) {
  int dev = 0;
  cudaError_t ce = cudaGetDevice(&dev);
  if (ce != cudaSuccess)
    return fail(RESHARD_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(ce));
  return occupancy(dev, 4, 0, 0, blocks_per_sm);
}

static reshard_status_t launch_tiles(const reshard_plan_s* plan, const Program& prog,
                                unsigned char* const* bufs, int nbufs, void* stream) {
  const int64_t total = prog.total_units();
  if (total == 0) return RESHARD_OK;
  if (nbufs > RESHARD_MAX_EXEC_BUFFERS) return fail(RESHARD_ERR_UNSUPPORTED, "too many buffers");
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev != plan->device)
    return fail(RESHARD_ERR_INVALID_ARG, "current device differs from the plan's device");

  const Dispatch d = decide(prog, bufs, nbufs, true);
  KernelParams kp;
  kp.tiles = prog.d_tiles;
  kp.prefix = prog.d_prefix;
  kp.goff = prog.d_goff;
  kp.gbuf = prog.d_gbuf;
  kp.total_units = total;
  kp.ntiles = int32_t(prog.tiles.size());
  kp.nbufs = nbufs;
  for (int i = 0; i < nbufs; ++i) kp.bufs[i] = bufs[i];
  for (int i = nbufs; i < RESHARD_MAX_EXEC_BUFFERS; ++i) kp.bufs[i] = nullptr;
  kp.flags = d.flags;
  kp.pad = 0;

  // A fully 16-byte-aligned fan-out goes through the TMA-staged pipeline.
  if (d.path == RESHARD_PATH_TMA_FANOUT) return launch_fanout_staged(plan, kp, prog, stream);
  if (d.kidx == kStagedRealign)
    return launch_realign_staged(plan->num_sms, kp, prog, stream);

  const int planes = prog.has_planes ? 1 : 0;
  const int kidx = d.kidx;
  int bps = 1;
  reshard_status_t st = occupancy(dev, kidx, planes, d.narrow, &bps);
  if (st != RESHARD_OK) return st;
  const int64_t max_grid = int64_t(plan->num_sms) * bps;
  const unsigned grid = unsigned(total < max_grid ? total : max_grid);
  void* args[] = {&kp};
  cudaError_t ce = cudaLaunchKernel(reinterpret_cast<const void*>(kKernels[d.narrow][kidx][planes]),
                                    dim3(grid), dim3(kThreads), args, 0,
                                    static_cast<cudaStream_t>(stream));
  if (ce != cudaSuccess)
    return fail(RESHARD_ERR_CUDA, std::string("kernel launch: ") + cudaGetErrorString(ce));
  return RESHARD_OK;
}


// Launch one program whose tables live at caller-given device addresses (the
// allocation-free entry point keeps them in a static device array).  Same kernel
// and grid rule as launch_program; needs no uploaded plan.
reshard_status_t launch_program(const reshard_plan_s* plan, const Program& prog,
                                unsigned char* const* bufs, int nbufs, void* stream) {
  reshard_status_t st = launch_tiles(plan, prog, bufs, nbufs, stream);
  if (st != RESHARD_OK || prog.tblocks.empty()) return st;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev != plan->device)
    return fail(RESHARD_ERR_INVALID_ARG, "current device differs from the plan's device");
  const uint32_t flags = destinations_congruent(prog, bufs) ? kFlagDstCongruent : 0u;
  return launch_transposes(plan, prog, bufs, nbufs, flags, stream);
}

reshard_status_t launch_fanout(const reshard_plan_s* plan, unsigned char* const* bufs, int nbufs,
                               void* stream) {
  reshard_status_t st = launch_program(plan, plan->prog[RESHARD_PROGRAM_FANOUT], bufs, nbufs, stream);
  if (st != RESHARD_OK) return st;
  return launch_program(plan, plan->prog[RESHARD_PROGRAM_REPLICATE], bufs, nbufs, stream);
}

reshard_status_t launch_program_tables(const Program& prog, const reshard_tile_t* d_tiles,
                                       const int64_t* d_prefix, const uint32_t* d_goff,
                                       const uint16_t* d_gbuf, int num_sms,
                                       unsigned char* const* bufs, int nbufs, void* stream) {
  // tables at explicit addresses carry tiles only: a program with transpose
  // blocks would leave the regions those blocks cover unwritten
  if (!prog.tblocks.empty())
    return fail(RESHARD_ERR_UNSUPPORTED, "program with transpose blocks at explicit table addresses");
  const int64_t total = prog.total_units();
  if (total == 0) return RESHARD_OK;
  if (nbufs > RESHARD_MAX_EXEC_BUFFERS) return fail(RESHARD_ERR_UNSUPPORTED, "too many buffers");
  int dev = -1;
  cudaError_t ce = cudaGetDevice(&dev);
  if (ce != cudaSuccess)
    return fail(RESHARD_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(ce));
  const Dispatch d = decide(prog, bufs, nbufs, false);
  const int planes = prog.has_planes ? 1 : 0;
  const int kidx = d.kidx;
  int bps = 1;
  if (kidx >= 0) {
    reshard_status_t st = occupancy(dev, kidx, planes, d.narrow, &bps);
    if (st != RESHARD_OK) return st;
  }

  KernelParams kp;
  kp.tiles = d_tiles;
  kp.prefix = d_prefix;
  kp.goff = d_goff;
  kp.gbuf = d_gbuf;
  kp.total_units = total;
  kp.ntiles = int32_t(prog.tiles.size());
  kp.nbufs = nbufs;
  for (int i = 0; i < nbufs; ++i) kp.bufs[i] = bufs[i];
  for (int i = nbufs; i < RESHARD_MAX_EXEC_BUFFERS; ++i) kp.bufs[i] = nullptr;
  kp.flags = d.flags;
  kp.pad = 0;
  if (kidx == kStagedRealign) return launch_realign_staged(num_sms, kp, prog, stream);

  const int64_t max_grid = int64_t(num_sms) * bps;
  const unsigned grid = unsigned(total < max_grid ? total : max_grid);
  void* args[] = {&kp};
  ce = cudaLaunchKernel(reinterpret_cast<const void*>(kKernels[d.narrow][kidx][planes]), dim3(grid),
                        dim3(kThreads), args, 0, static_cast<cudaStream_t>(stream));
  if (ce != cudaSuccess)
    return fail(RESHARD_ERR_CUDA, std::string("kernel launch: ") + cudaGetErrorString(ce));
  return RESHARD_OK;
}

}  // namespace rs
