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
// issues kUnroll independent loads before it stores, and each loaded vector is
// stored to every destination buffer of the tile's group (the fan-out: the
// source region is read from HBM once, written R times).  Loads and stores use
// the evict-first (streaming) cache policy because no byte is touched twice.
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

namespace rs {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;

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

template <typename T>
__device__ __forceinline__ T load_stream(const unsigned char* p) {
  return __ldcs(reinterpret_cast<const T*>(p));
}
template <typename T>
__device__ __forceinline__ void store_stream(unsigned char* p, const T& v) {
  __stcs(reinterpret_cast<T*>(p), v);
}

// Bytes [0, nbytes) of a contiguous run: from src to dst + dofs for each of
// the R destination buffers dst in sdst.
template <int W>
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
// streamed one at a time by the whole CTA; shorter rows are packed
// kThreads / vpr to a pass, one thread per vector, and every thread carries
// kUnroll rows at once.
template <int W, bool PLANES>
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
#pragma unroll 1
    for (uint32_t row = r_begin; row < r_end; ++row)
      copy_run<W>(s0 + src_row(row), sdst, R, t.dst_off + dst_row(row), t.row_bytes);
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

template <int W, bool PLANES>
__global__ void __launch_bounds__(kThreads, PLANES ? 2 : 4)
    reshard_copy_kernel(const __grid_constant__ KernelParams p) {
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
      copy_run<W>(src + t.src_off + b0, s_dst, R, t.dst_off + b0, uint32_t(b1 - b0));
    } else {
      const uint32_t upr = t.row_bytes >= kUnitBytes ? 1u : uint32_t(kUnitBytes) / t.row_bytes;
      const uint64_t rows = uint64_t(t.nrows) * t.nplanes;
      const uint32_t r_begin = uint32_t(a * upr);
      const uint32_t r_end = uint32_t(min(uint64_t(b) * upr, rows));
      if (PLANES && t.nplanes > 1) copy_rows<W, true>(t, src, s_dst, R, r_begin, r_end);
      else copy_rows<W, false>(t, src, s_dst, R, r_begin, r_end);
    }
    u0 = tb + b;
    ++ti;
  }
}


using KernelFn = void (*)(KernelParams);

// Instantiations indexed by [log2 W][planes].
const KernelFn kKernels[5][2] = {
    {reshard_copy_kernel<1, false>, reshard_copy_kernel<1, true>},
    {reshard_copy_kernel<2, false>, reshard_copy_kernel<2, true>},
    {reshard_copy_kernel<4, false>, reshard_copy_kernel<4, true>},
    {reshard_copy_kernel<8, false>, reshard_copy_kernel<8, true>},
    {reshard_copy_kernel<16, false>, reshard_copy_kernel<16, true>},
};

std::mutex g_occ_mu;
std::map<std::pair<int, int>, int> g_occ;  // (device, kernel index) -> blocks per SM

reshard_status_t occupancy(int device, int w_log2, int planes, int* blocks) {
  const std::pair<int, int> key(device, w_log2 * 2 + planes);
  std::lock_guard<std::mutex> lk(g_occ_mu);
  auto it = g_occ.find(key);
  if (it != g_occ.end()) {
    *blocks = it->second;
    return RESHARD_OK;
  }
  int n = 0;
  cudaError_t ce = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
      &n, reinterpret_cast<const void*>(kKernels[w_log2][planes]), kThreads, 0);
  if (ce != cudaSuccess)
    return fail(RESHARD_ERR_CUDA, std::string("occupancy query: ") + cudaGetErrorString(ce));
  n = n > 0 ? n : 1;
  g_occ[key] = n;
  *blocks = n;
  return RESHARD_OK;
}

}  // namespace

reshard_status_t copy_kernel_occupancy(int* blocks_per_sm) {
  int dev = 0;
  cudaError_t ce = cudaGetDevice(&dev);
  if (ce != cudaSuccess)
    return fail(RESHARD_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(ce));
  return occupancy(dev, 4, 0, blocks_per_sm);
}

reshard_status_t launch_program(const reshard_plan_s* plan, const Program& prog,
                                unsigned char* const* bufs, int nbufs, void* stream) {
  const int64_t total = prog.total_units();
  if (total == 0) return RESHARD_OK;
  if (nbufs > RESHARD_MAX_EXEC_BUFFERS) return fail(RESHARD_ERR_UNSUPPORTED, "too many buffers");
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev != plan->device)
    return fail(RESHARD_ERR_INVALID_ARG, "current device differs from the plan's device");

  // Widest access every tile of the program allows with these buffers.
  uint64_t align = prog.align_bits;
  for (int i = 0; i < nbufs; ++i) align |= reinterpret_cast<uint64_t>(bufs[i]);
  int w_log2 = 4;
  while (w_log2 > 0 && (align & ((uint64_t(1) << w_log2) - 1)) != 0) --w_log2;
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

  // A fully 16-byte-aligned fan-out goes through the TMA-staged pipeline.
  if (prog.staged && w_log2 == 4) return launch_fanout_staged(plan, kp, stream);

  const int planes = prog.has_planes ? 1 : 0;
  int bps = 1;
  reshard_status_t st = occupancy(dev, w_log2, planes, &bps);
  if (st != RESHARD_OK) return st;
  const int64_t max_grid = int64_t(plan->num_sms) * bps;
  const unsigned grid = unsigned(total < max_grid ? total : max_grid);
  void* args[] = {&kp};
  cudaError_t ce = cudaLaunchKernel(reinterpret_cast<const void*>(kKernels[w_log2][planes]),
                                    dim3(grid), dim3(kThreads), args, 0,
                                    static_cast<cudaStream_t>(stream));
  if (ce != cudaSuccess)
    return fail(RESHARD_ERR_CUDA, std::string("kernel launch: ") + cudaGetErrorString(ce));
  return RESHARD_OK;
}


// Launch one program whose tables live at caller-given device addresses (the
// allocation-free entry point keeps them in a static device array).  Same kernel
// and grid rule as launch_program; needs no uploaded plan.
reshard_status_t launch_program_tables(const Program& prog, const reshard_tile_t* d_tiles,
                                       const int64_t* d_prefix, const uint32_t* d_goff,
                                       const uint16_t* d_gbuf, int num_sms,
                                       unsigned char* const* bufs, int nbufs, void* stream) {
  const int64_t total = prog.total_units();
  if (total == 0) return RESHARD_OK;
  if (nbufs > RESHARD_MAX_EXEC_BUFFERS) return fail(RESHARD_ERR_UNSUPPORTED, "too many buffers");
  int dev = -1;
  cudaError_t ce = cudaGetDevice(&dev);
  if (ce != cudaSuccess)
    return fail(RESHARD_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(ce));
  uint64_t align = prog.align_bits;
  for (int i = 0; i < nbufs; ++i) align |= reinterpret_cast<uint64_t>(bufs[i]);
  int w_log2 = 4;
  while (w_log2 > 0 && (align & ((uint64_t(1) << w_log2) - 1)) != 0) --w_log2;
  const int planes = prog.has_planes ? 1 : 0;
  int bps = 1;
  reshard_status_t st = occupancy(dev, w_log2, planes, &bps);
  if (st != RESHARD_OK) return st;

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

  const int64_t max_grid = int64_t(num_sms) * bps;
  const unsigned grid = unsigned(total < max_grid ? total : max_grid);
  void* args[] = {&kp};
  ce = cudaLaunchKernel(reinterpret_cast<const void*>(kKernels[w_log2][planes]), dim3(grid),
                        dim3(kThreads), args, 0, static_cast<cudaStream_t>(stream));
  if (ce != cudaSuccess)
    return fail(RESHARD_ERR_CUDA, std::string("kernel launch: ") + cudaGetErrorString(ce));
  return RESHARD_OK;
}

}  // namespace rs
