// transpose.cu -- transpose blocks: narrow innermost pieces regrouped by rows (sm_103a).
//
// A block covers nrows consecutive rows of row_bytes on the wide side (one
// contiguous range of one buffer, or of every buffer of one destination group)
// and seg_count narrow segments, each a dense nrows x width range of its own
// buffer (or destination group) that fills bytes [col, col + width) of every
// wide row.  A CTA takes a contiguous share of the program's blocks and, per
// block:
//   gather  (narrow sources -> wide destination group): copies every segment
//           into its columns of a shared-memory image of the rows, then writes
//           the image with 16-byte stores to every replica;
//   scatter (wide source -> narrow destination groups): loads the rows with
//           16-byte loads, then writes every segment to its replicas.
// The shared-memory image is shifted by the wide side's address mod 16, so its
// 16-byte vectors line up with aligned global addresses.  Narrow-side copies
// move elements of U bytes (the widest unit every address, width and column of
// the block allows), walking each segment's dense range in order, so both
// sides of every copy are coalesced.
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
// staging area for the narrow side: every segment's dense range in whole 16-byte
// granules (at most one extra granule per segment)
constexpr int kStageBytes = int(kTransposeBlockBytes) + 32 * int(kTransposeMaxSegs) + 64;
constexpr int kDynSmem = kImageBytes + kStageBytes;
constexpr int kMaxReplicaPtrs = int(kTransposeMaxReplicaPtrs);

struct TransposeParams {
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
  uint32_t gstart;           // first staging granule of the segment
  uint32_t gmis;             // narrow global address mod 16 (replica 0 for scatter)
  uint32_t nbytes;           // width * nrows
};

template <int U> struct UType;
template <> struct UType<1> { using T = uint8_t; };
template <> struct UType<2> { using T = uint16_t; };
template <> struct UType<4> { using T = uint32_t; };
template <> struct UType<8> { using T = uint2; };

// segment owning staging granule g (largest k with gstart[k] <= g)
__device__ __forceinline__ int find_granule(const SegInfo* si, int K, uint32_t g) {
  int lo = 0, hi = K - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (si[mid].gstart <= g) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// gather, phase 1a: every segment's dense source range -> staging, as whole aligned
// 16-byte granules (granule j of segment k at staging byte 16 (gstart_k + j))
__device__ __forceinline__ void gather_stage(const SegInfo* si, int K, uint32_t ngran,
                                             unsigned char* stg) {
#pragma unroll 1
  for (uint32_t g0 = threadIdx.x; g0 < ngran; g0 += kTThreads * kTVecUnroll) {
    uint4 v[kTVecUnroll];
#pragma unroll
    for (int j = 0; j < kTVecUnroll; ++j) {
      const uint32_t g = g0 + j * kTThreads;
      if (g < ngran) {
        const SegInfo& s = si[find_granule(si, K, g)];
        v[j] = __ldcs(reinterpret_cast<const uint4*>(s.src - s.gmis + 16 * size_t(g - s.gstart)));
      }
    }
#pragma unroll
    for (int j = 0; j < kTVecUnroll; ++j) {
      const uint32_t g = g0 + j * kTThreads;
      if (g < ngran) *reinterpret_cast<uint4*>(stg + 16 * size_t(g)) = v[j];
    }
  }
}

// gather, phase 1b: staging -> columns of the image (shared memory only), one
// warp per segment, lanes over its elements
template <int U>
__device__ __forceinline__ void gather_place(const SegInfo* si, int K, uint32_t nr,
                                             const unsigned char* stg, unsigned char* img,
                                             uint32_t mis, uint32_t L) {
  using T = typename UType<U>::T;
  const int warp = int(threadIdx.x >> 5), lane = int(threadIdx.x & 31);
  for (int k = warp; k < K; k += kTThreads / 32) {
    const SegInfo& s = si[k];
    const uint32_t n = s.units * nr;
    const unsigned char* from = stg + 16 * s.gstart + s.gmis;
    unsigned char* to = img + mis + s.col;
#pragma unroll 4
    for (uint32_t local = lane; local < n; local += 32) {
      const uint32_t row = fastdiv(local, s.m, s.l);
      const uint32_t c = local - row * s.units;
      *reinterpret_cast<T*>(to + row * L + c * U) = *reinterpret_cast<const T*>(from + local * U);
    }
  }
}

// scatter, phase 2a: image columns -> staging, laid out so that every segment's
// destination range (replica 0) falls on whole 16-byte granules; warp per segment
template <int U>
__device__ __forceinline__ void scatter_stage(const SegInfo* si, int K, uint32_t nr,
                                              const unsigned char* img, uint32_t mis, uint32_t L,
                                              unsigned char* stg) {
  using T = typename UType<U>::T;
  const int warp = int(threadIdx.x >> 5), lane = int(threadIdx.x & 31);
  for (int k = warp; k < K; k += kTThreads / 32) {
    const SegInfo& s = si[k];
    const uint32_t n = s.units * nr;
    const unsigned char* from = img + mis + s.col;
    unsigned char* to = stg + 16 * s.gstart + s.gmis;
#pragma unroll 4
    for (uint32_t local = lane; local < n; local += 32) {
      const uint32_t row = fastdiv(local, s.m, s.l);
      const uint32_t c = local - row * s.units;
      *reinterpret_cast<T*>(to + local * U) = *reinterpret_cast<const T*>(from + row * L + c * U);
    }
  }
}

// scatter, phase 2b: staging granules -> every replica of every segment, warp per
// segment; whole granules of replicas aligned like replica 0 go out as 16-byte stores
__device__ __forceinline__ void scatter_write(const SegInfo* si, int K, const unsigned char* stg,
                                              unsigned char* const* ptrs) {
  const int warp = int(threadIdx.x >> 5), lane = int(threadIdx.x & 31);
  for (int k = warp; k < K; k += kTThreads / 32) {
    const SegInfo& s = si[k];
    const uint32_t end = s.gmis + s.nbytes;      // segment end, granule-relative bytes
    const uint32_t ng = (end + 15u) >> 4;
    for (uint32_t j = lane; j < ng; j += 32) {
      const uint32_t lo = j == 0 ? s.gmis : 0u;
      const uint32_t hi = min(16u, end - 16u * j);
      const unsigned char* src = stg + 16 * size_t(s.gstart + j);
      const uint4 v = *reinterpret_cast<const uint4*>(src);
      for (uint32_t r = 0; r < s.rcnt; ++r) {
        unsigned char* base = ptrs[s.rbeg + r] + s.off;  // segment byte 0 of this replica
        if ((reinterpret_cast<uintptr_t>(base) & 15u) == s.gmis) {
          // aligned like replica 0: whole granules in one store, partial ones in the
          // widest aligned stores that fit
          unsigned char* g = base - s.gmis + 16 * size_t(j);
          if (lo == 0 && hi == 16) __stcs(reinterpret_cast<uint4*>(g), v);
          else staging::store_partial16(g, v, lo, hi);
        } else {
          for (uint32_t b = lo; b < hi; ++b) base[16 * j + b - s.gmis] = src[b];
        }
      }
    }
  }
}

__global__ void __launch_bounds__(kTThreads, 4)
    reshard_transpose_kernel(const __grid_constant__ TransposeParams p) {
  extern __shared__ __align__(16) unsigned char dyn[];
  unsigned char* img = dyn;                // wide rows, shifted by the wide address mod 16
  unsigned char* stg = dyn + kImageBytes;  // narrow ranges in whole 16-byte granules
  __shared__ SegInfo si[kTransposeMaxSegs];
  __shared__ unsigned char* ptrs[kMaxReplicaPtrs];
  __shared__ unsigned int s_align;
  __shared__ uint32_t s_ngran;
  const bool congruent = (p.flags & kFlagDstCongruent) != 0;
  const int64_t b0 = p.nblocks * int64_t(blockIdx.x) / int64_t(gridDim.x);
  const int64_t b1 = p.nblocks * int64_t(blockIdx.x + 1) / int64_t(gridDim.x);
  for (int64_t bi = b0; bi < b1; ++bi) {
    const reshard_tblock_t blk = p.blocks[bi];
    const uint32_t L = blk.row_bytes, nr = blk.nrows, K = blk.seg_count;
    const uint32_t n = L * nr;
    const bool gather = blk.direction == 0;
    __syncthreads();  // the previous block is completely done with img/si/ptrs
    // wide-side pointers: gather -> the destination group in ptrs[0..R); scatter -> source
    int R = 0;
    const unsigned char* wsrc = nullptr;
    if (gather) {
      const uint32_t g0 = p.goff[blk.wide];
      R = int(p.goff[blk.wide + 1] - g0);
      for (int i = threadIdx.x; i < R; i += kTThreads) ptrs[i] = p.bufs[p.gbuf[g0 + i]];
    } else {
      wsrc = p.bufs[blk.wide] + blk.wide_off;
    }
    __syncthreads();
    const uint32_t mis = gather ? uint32_t(reinterpret_cast<uintptr_t>(ptrs[0] + blk.wide_off) & 15u)
                                : uint32_t(reinterpret_cast<uintptr_t>(wsrc) & 15u);
    if (threadIdx.x == 0) s_align = L | 8u;
    __syncthreads();
    // per-segment set-up (one thread per segment), alignment of every narrow access
    for (uint32_t k = threadIdx.x; k < K; k += kTThreads) {
      const reshard_tseg_t sg = p.segs[blk.seg_begin + k];
      unsigned int a = sg.width | (mis + sg.col);
      if (gather) {
        si[k].src = p.bufs[sg.narrow] + sg.narrow_off;
        si[k].gmis = unsigned(reinterpret_cast<uintptr_t>(si[k].src) & 15u);
        a |= unsigned(reinterpret_cast<uintptr_t>(si[k].src));
      } else {
        si[k].off = sg.narrow_off;
        const uint32_t g0 = p.goff[sg.narrow];
        const uint32_t rc = p.goff[sg.narrow + 1] - g0;
        si[k].rcnt = rc;
        si[k].gmis =
            unsigned(reinterpret_cast<uintptr_t>(p.bufs[p.gbuf[g0]] + sg.narrow_off) & 15u);
        a |= si[k].gmis;
      }
      si[k].nbytes = sg.width * nr;
      si[k].col = sg.col;
      si[k].units = sg.width;  // bytes for now
      atomicOr(&s_align, a);
    }
    __syncthreads();
    const unsigned int al = s_align;
    const uint32_t U = (al & 1u) ? 1u : (al & 2u) ? 2u : (al & 4u) ? 4u : 8u;
    if (threadIdx.x < 32) {
      // staging granules and replica pointer slots, exclusive prefix in segment order:
      // each lane owns segments [4 lane, 4 lane + 4) (K <= 128), then a warp scan
      const int lane = int(threadIdx.x);
      uint32_t rc[4], gc[4], rsum = 0, gsum = 0;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t k = uint32_t(4 * lane + q);
        rc[q] = (k < K && !gather) ? si[k].rcnt : 0u;
        gc[q] = k < K ? (si[k].gmis + si[k].nbytes + 15u) >> 4 : 0u;
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
          si[k].units /= U;
          si[k].rbeg = rb;
          si[k].gstart = gs;
        }
        rb += rc[q];
        gs += gc[q];
      }
      if (lane == 31) s_ngran = ginc;
    }
    __syncthreads();
    for (uint32_t k = threadIdx.x; k < K; k += kTThreads) {
      fastdiv_init(si[k].units, &si[k].m, &si[k].l);
      if (!gather) {
        const reshard_tseg_t sg = p.segs[blk.seg_begin + k];
        const uint32_t g0 = p.goff[sg.narrow];
        for (uint32_t r = 0; r < si[k].rcnt; ++r) ptrs[si[k].rbeg + r] = p.bufs[p.gbuf[g0 + r]];
      }
    }
    __syncthreads();
    const uint32_t ngran = s_ngran;

    if (gather) {
      gather_stage(si, int(K), ngran, stg);
      __syncthreads();
      switch (U) {
        case 1: gather_place<1>(si, int(K), nr, stg, img, mis, L); break;
        case 2: gather_place<2>(si, int(K), nr, stg, img, mis, L); break;
        case 4: gather_place<4>(si, int(K), nr, stg, img, mis, L); break;
        default: gather_place<8>(si, int(K), nr, stg, img, mis, L); break;
      }
      __syncthreads();
      // image [mis, mis + n) -> each replica's [wide_off, wide_off + n)
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
        for (uint32_t k = threadIdx.x; k < m16; k += kTThreads)
          __stcs(reinterpret_cast<uint4*>(d + h + 16 * k),
                 *reinterpret_cast<const uint4*>(img + mis + h + 16 * k));
        for (uint32_t i = h + 16 * m16 + threadIdx.x; i < n; i += kTThreads) d[i] = img[mis + i];
      }
    } else {
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
      switch (U) {
        case 1: scatter_stage<1>(si, int(K), nr, img, mis, L, stg); break;
        case 2: scatter_stage<2>(si, int(K), nr, img, mis, L, stg); break;
        case 4: scatter_stage<4>(si, int(K), nr, img, mis, L, stg); break;
        default: scatter_stage<8>(si, int(K), nr, img, mis, L, stg); break;
      }
      __syncthreads();
      scatter_write(si, int(K), stg, ptrs);
    }
  }
}

std::mutex g_t_mu;
std::map<int, int> g_t_occ;  // device -> blocks per SM

}  // namespace

reshard_status_t launch_transposes(const reshard_plan_s* plan, const Program& prog,
                                   unsigned char* const* bufs, int nbufs, uint32_t flags,
                                   void* stream) {
  if (prog.tblocks.empty()) return RESHARD_OK;
  int dev = -1;
  cudaError_t ce = cudaGetDevice(&dev);
  if (ce != cudaSuccess)
    return fail(RESHARD_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(ce));
  int bps = 0;
  {
    std::lock_guard<std::mutex> lk(g_t_mu);
    auto it = g_t_occ.find(dev);
    if (it == g_t_occ.end()) {
      ce = cudaFuncSetAttribute(reinterpret_cast<const void*>(reshard_transpose_kernel),
                                cudaFuncAttributeMaxDynamicSharedMemorySize, kDynSmem);
      if (ce == cudaSuccess)
        ce = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
            &bps, reinterpret_cast<const void*>(reshard_transpose_kernel), kTThreads, kDynSmem);
      if (ce != cudaSuccess)
        return fail(RESHARD_ERR_CUDA, std::string("transpose kernel set-up: ") + cudaGetErrorString(ce));
      bps = bps > 0 ? bps : 1;
      g_t_occ[dev] = bps;
    } else {
      bps = it->second;
    }
  }
  TransposeParams tp;
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
  ce = cudaLaunchKernel(reinterpret_cast<const void*>(reshard_transpose_kernel), dim3(grid),
                        dim3(kTThreads), args, kDynSmem, static_cast<cudaStream_t>(stream));
  if (ce != cudaSuccess)
    return fail(RESHARD_ERR_CUDA, std::string("kernel launch: ") + cudaGetErrorString(ce));
  return RESHARD_OK;
}

}  // namespace rs
