// realign_staged.cu -- TMA-staged copy for programs whose offsets, strides, row
// lengths or buffers are not all 16-byte aligned (sm_103a).
//
// Each CTA runs three roles over pieces of consecutive work units that it takes
// from a per-launch work queue as it goes (CTAs on faster SMs take more), in
// chunks of one tile each; the producer hands every chunk to the other roles
// through a descriptor beside its stage:
//   warp 0, the producer, copies the aligned 16-byte granules that hold the
//     chunk's source bytes into an input stage -- one cp.async.bulk copy for a
//     piece of a run, of a long row, or of rows that follow one another in the
//     source; otherwise every row into its own slot, with one bulk copy per
//     long row or 16-byte cp.async copies for short ones -- completion counted
//     on the stage's "full" mbarrier (bytes for bulk copies, the lanes' copies
//     for cp.async), and records each row's destination offset and stage
//     position in the stage's row table;
//   kConsumerWarps consumer warps cover every destination granule (16 aligned
//     destination bytes) of every row with one thread, cutting the granule's
//     bytes out of five aligned 4-byte stage words with funnel shifts;
//   by default each consumer writes its granules to every replica itself
//     with aligned 16-byte stores (one realignment when every destination
//     buffer has the same address mod 16, one per replica otherwise; the
//     partial first and last granule of a row with the widest aligned stores
//     that fit);
//   with kFlagBulkStores (wide fan-outs to destinations that share their
//     address mod 16) the whole granules go instead to an output stage that
//     mirrors the destinations' alignment, and the store warp writes each row's
//     whole granules to every replica with cp.async.bulk stores.
// Source bytes cross HBM once; bytes of the aligned source granules outside
// the chunk are read into the stage and never written anywhere.  No multicast
// is used.
//
// Every mbarrier wait is bounded; a wait that runs out records a code in the
// device status word and the warp returns after waiting (boundedly) for the
// bulk copies it issued.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>
#include <string>

#include "internal.h"
#include "staging.cuh"

namespace rs {
namespace {

using namespace staging;

// Row slot slack: 16 bytes ahead of the granules for a negative shift and room
// behind them for the second word of the last granule.
constexpr uint32_t kPad = 80;
constexpr uint32_t kHead = 16;  // a stage's first granule lands here
constexpr int kStages = 3;      // input stages
constexpr int kConsumerWarps = 8;
// Rows that are neither contiguous with their neighbours in the source nor at
// least this long are staged with cp.async (a bulk copy each costs the copy
// engine about as long as 1 KB of streaming).
constexpr uint32_t kCpAsyncRowBytes = 2048;
constexpr int kConsumerThreads = 32 * kConsumerWarps;

// BULK = false: consumers store; BULK = true: output stages and a store warp.
template <bool BULK>
struct Config {
  // three output stages (two were 1-2% slower on fan-outs to 20-34 replicas, where a
  // stage waits for all of its bulk stores to read it; a third costs no occupancy)
  static constexpr int kOutStages = BULK ? 3 : 0;
  static constexpr uint32_t kStageBytes = BULK ? 16 * 1024 : 20 * 1024;
  static constexpr int kStoreWarp = 1 + kConsumerWarps;
  static constexpr int kThreads = 32 * (1 + kConsumerWarps + (BULK ? 1 : 0));
  static constexpr int kDynSmem = (kStages + kOutStages) * int(kStageBytes);
  using Walker = ChunkWalker<kStageBytes, kPad>;
  static constexpr uint32_t kMaxRows = Walker::kMaxRows;
};

// Destination granule k of a row whose first destination byte sits dmis bytes
// into its granule and whose first source byte is staged at stage + spos.
// Byte j of the granule is row byte 16k + j - dmis, staged at
// stage + spos - dmis + 16k + j (spos >= kHead, so the start is in the stage).
// The granule is five aligned 4-byte stage words funnel-shifted by the byte
// offset (no run-time word selection; the reads stay inside the 32 bytes from
// the aligned 16 bytes that hold its first byte).
__device__ __forceinline__ uint4 granule(const unsigned char* stage, uint32_t spos, uint32_t dmis,
                                         uint32_t k) {
  const uint32_t at = spos - dmis + 16u * k;
  const uint32_t* w = reinterpret_cast<const uint32_t*>(stage + (at & ~3u));
  const uint32_t sh = 8u * (at & 3u);
  const uint32_t w0 = w[0], w1 = w[1], w2 = w[2], w3 = w[3], w4 = sh ? w[4] : 0u;
  return make_uint4(__funnelshift_r(w0, w1, sh), __funnelshift_r(w1, w2, sh),
                    __funnelshift_r(w2, w3, sh), __funnelshift_r(w3, w4, sh));
}

// Granule k (bytes v) of a row to one replica: dst + doff is the row's first
// destination byte.
__device__ __forceinline__ void put_granule(unsigned char* dst, int64_t doff, uint32_t dmis,
                                            uint32_t n, uint32_t G, uint32_t k, const uint4& v) {
  unsigned char* g = dst + doff - int64_t(dmis) + 16 * int64_t(k);
  uint32_t lo, hi;
  granule_span(dmis, n, G, k, &lo, &hi);
  if (lo == 0 && hi == 16) __stcs(reinterpret_cast<uint4*>(g), v);
  else store_partial16(g, v, lo, hi);
}

// A wait by the whole warp, with one answer for all lanes.  Every lane polls:
// a wait left to one lane of a diverged warp was measured to return late.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, kWaitPolls)) != 0;
}

// BULK requires every destination buffer at the same address mod 16.
template <bool BULK>
__global__ void __launch_bounds__(Config<BULK>::kThreads)
    realign_staged_kernel(const __grid_constant__ KernelParams p, unsigned int* status,
                          unsigned int* queue, const PieceSchedule sched) {
  using C = Config<BULK>;
  using Walker = typename C::Walker;
  constexpr uint32_t kStageBytes = C::kStageBytes;
  constexpr int kOutStages = C::kOutStages > 0 ? C::kOutStages : 1;
  constexpr int kStoreWarp = C::kStoreWarp;
  constexpr uint32_t kMaxRows = C::kMaxRows;
  extern __shared__ __align__(1024) unsigned char stage_mem[];
  __shared__ __align__(8) uint64_t full[kStages], empty[kStages];
  __shared__ __align__(8) uint64_t out_full[kOutStages], out_free[kOutStages];
  __shared__ int64_t row_doff[kStages][kMaxRows];
  __shared__ uint16_t row_spos[kStages][kMaxRows];
  __shared__ unsigned char* dst_ptr[kStages][kMaxGroup];
  __shared__ StageDesc desc[kStages];
  // the chunk's row length and replica count, from the producer: the consumers and
  // the store warp read no tile record or group table from global memory
  __shared__ uint32_t desc_len[kStages], desc_R[kStages];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // bulk: the store warp writes whole granules from the output stages and
  // releases the input stages; otherwise the consumers write everything and
  // release them
  const bool congruent = (p.flags & kFlagDstCongruent) != 0;
  constexpr bool bulk = BULK;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], bulk ? 1u : uint32_t(kConsumerWarps));
    }
    for (int o = 0; o < C::kOutStages; ++o) {
      mbar_init(&out_full[o], kConsumerWarps);
      mbar_init(&out_free[o], 1);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  unsigned char* const in_mem = stage_mem;
  unsigned char* const out_mem = stage_mem + size_t(kStages) * kStageBytes;
  uint32_t n = 0;
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    Walker w;
    Chunk c;
    int stage_tile[kStages];
    for (int s = 0; s < kStages; ++s) stage_tile[s] = -1;
    int cur_tile = -1;
    uint32_t g0 = 0, R = 0;  // the current tile's destination group
    bool ok = true;
    const int64_t npieces = sched.count();
    uint32_t piece = grab_piece(queue, lane);
    while (ok && int64_t(piece) < npieces) {
    const uint32_t next_piece = grab_piece(queue, lane);  // asked early, used later
    int64_t u0, u1;
    sched.range(piece, &u0, &u1);
    w.start_range(&p, u0, u1);
    while (w.next(&c)) {
      const int s = int(n % kStages);
      if (n >= uint32_t(kStages) && !warp_wait(&empty[s], ((n / kStages) - 1) & 1u)) {
        if (lane == 0) atomicExch(status, kStatusProducerWait);
        ok = false;
        break;
      }
      const reshard_tile_t& t = w.t;
      if (c.ti != cur_tile) {
        g0 = p.goff[t.dst_group];
        R = p.goff[t.dst_group + 1] - g0;
        cur_tile = c.ti;
      }
      const uint32_t nr = c.kind == 1 ? uint32_t(c.b - c.a) : 1u;
      const uint32_t len = c.kind == 1 ? t.row_bytes : c.bytes;
      if (lane == 0) {
        desc[s] = StageDesc{c.ti, c.kind, c.bytes, c.a, c.b};
        desc_len[s] = len;
        desc_R[s] = R;
      }
      if (stage_tile[s] != c.ti) {
        // the stage's destination pointers (the stage's last readers are done)
        for (uint32_t i = lane; i < R; i += 32) dst_ptr[s][i] = p.bufs[p.gbuf[g0 + i]];
        stage_tile[s] = c.ti;
      }
      const unsigned char* src = p.bufs[t.src_buf];
      unsigned char* stage = in_mem + size_t(s) * kStageBytes;
      if (c.kind != 1 || Walker::source_contiguous(t)) {
        // one copy: the chunk's bytes are contiguous in the source
        const unsigned char* sa = c.kind == 0   ? src + t.src_off + c.a
                                  : c.kind == 1 ? src + src_row(t, c.a)
                                                : src + src_row(t, c.a) + c.b;
        const uintptr_t a = reinterpret_cast<uintptr_t>(sa);
        const uintptr_t lo = a & ~uintptr_t(15);
        const uintptr_t hi = (a + uintptr_t(nr) * len + 15u) & ~uintptr_t(15);
        for (uint32_t r = lane; r < nr; r += 32) {
          row_spos[s][r] = uint16_t(kHead + (a - lo) + r * len);
          row_doff[s][r] = c.kind == 0   ? t.dst_off + c.a
                           : c.kind == 1 ? dst_row(t, c.a + r)
                                         : dst_row(t, c.a) + c.b;
        }
        __syncwarp();
        if (lane == 0) {
          mbar_arrive_expect(&full[s], uint32_t(hi - lo));
          bulk_load(stage + kHead, reinterpret_cast<const void*>(lo), uint32_t(hi - lo), &full[s]);
        }
      } else if (len < kCpAsyncRowBytes) {
        // short rows, each into its own slot, in 16-byte cp.async copies by
        // all lanes (one lane per row): the full barrier's phase also waits
        // for every lane's copies
        const uint32_t slot = Walker::slot(len);
        for (uint32_t r = lane; r < nr; r += 32) {
          const uintptr_t a = reinterpret_cast<uintptr_t>(src + src_row(t, c.a + r));
          const uintptr_t lo = a & ~uintptr_t(15), hi = (a + len + 15u) & ~uintptr_t(15);
          unsigned char* d = stage + size_t(r) * slot + kHead;
          for (uintptr_t x = lo; x < hi; x += 16, d += 16)
            cp_async16(d, reinterpret_cast<const void*>(x));
          row_spos[s][r] = uint16_t(r * slot + kHead + (a & 15u));
          row_doff[s][r] = dst_row(t, c.a + r);
        }
        cp_async_arrive(&full[s]);
        __syncwarp();
        if (lane == 0) mbar_arrive(&full[s]);
      } else {
        // one bulk copy per row, each into its own slot
        const uint32_t slot = Walker::slot(len);
        uint32_t tx = 0;
        for (uint32_t r = lane; r < nr; r += 32) {
          const uintptr_t a = reinterpret_cast<uintptr_t>(src + src_row(t, c.a + r));
          tx += uint32_t(((a + len + 15u) & ~uintptr_t(15)) - (a & ~uintptr_t(15)));
          row_spos[s][r] = uint16_t(r * slot + kHead + (a & 15u));
          row_doff[s][r] = dst_row(t, c.a + r);
        }
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) tx += __shfl_xor_sync(0xffffffffu, tx, d);
        __syncwarp();
        if (lane == 0) mbar_arrive_expect(&full[s], tx);
        __syncwarp();
        for (uint32_t r = lane; r < nr; r += 32) {
          const uintptr_t a = reinterpret_cast<uintptr_t>(src + src_row(t, c.a + r));
          const uintptr_t lo = a & ~uintptr_t(15), hi = (a + len + 15u) & ~uintptr_t(15);
          bulk_load(stage + size_t(r) * slot + kHead, reinterpret_cast<const void*>(lo),
                    uint32_t(hi - lo), &full[s]);
        }
      }
      ++n;
    }
    piece = next_piece;
    }
    // end marker: a stage whose descriptor says "no more chunks", with no bytes
    if (ok) {
      const int s = int(n % kStages);
      if (n >= uint32_t(kStages) && !warp_wait(&empty[s], ((n / kStages) - 1) & 1u)) {
        if (lane == 0) atomicExch(status, kStatusProducerWait);
      } else {
        if (lane == 0) {
          desc[s].ti = -1;
          mbar_arrive(&full[s]);
        }
        ++n;
      }
    }
    // wait (boundedly) for the copies still landing in the stages
    const uint32_t issued = n;
    for (uint32_t m = issued > uint32_t(kStages) ? issued - kStages : 0u; m < issued; ++m)
      warp_wait(&full[m % kStages], (m / kStages) & 1u);
  } else if (warp < kStoreWarp) {
    // ------------------------------------------------------------ consumers
    const uint32_t ct = threadIdx.x - 32;
    while (true) {
      const int s = int(n % kStages), o = int(n % kOutStages);
      if (!warp_wait(&full[s], (n / kStages) & 1u) ||
          (bulk && n >= uint32_t(kOutStages) &&
           !warp_wait(&out_free[o], ((n / kOutStages) - 1) & 1u))) {
        if (lane == 0) atomicExch(status, kStatusConsumerWait);
        break;
      }
      const StageDesc c = desc[s];
      if (c.ti < 0) {
        // pass the end on to the store warp through the output stage's barrier
        if (bulk && lane == 0) mbar_arrive(&out_full[o]);
        break;
      }
      const int R = int(desc_R[s]);
      const uint32_t nr = c.kind == 1 ? uint32_t(c.b - c.a) : 1u;
      const uint32_t len = desc_len[s];
      const uint32_t gmax = (len + 30u) >> 4;  // granules a row of len bytes can touch
      const uint32_t ost = Walker::out_stride(len);
      const unsigned char* stage = in_mem + size_t(s) * kStageBytes;
      unsigned char* out = out_mem + size_t(o) * kStageBytes;
      unsigned char* const* dptr = dst_ptr[s];
      // granule k of staged row r; dmis and G are the first replica's (every
      // replica's on the bulk and congruent paths)
      auto item = [&](uint32_t r, uint32_t k, int64_t doff, uint32_t spos, uint32_t dmis,
                      uint32_t G) {
        if (bulk) {
          if (k >= G) return;
          const uint4 v = granule(stage, spos, dmis, k);
          uint32_t lo, hi;
          granule_span(dmis, len, G, k, &lo, &hi);
          if (lo == 0 && hi == 16) {
            *reinterpret_cast<uint4*>(out + size_t(r) * ost + 16u * k) = v;
          } else {
            for (int j = 0; j < R; ++j)
              store_partial16(dptr[j] + doff - int64_t(dmis) + 16 * int64_t(k), v, lo, hi);
          }
        } else if (congruent) {
          if (k >= G) return;
          const uint4 v = granule(stage, spos, dmis, k);
          uint32_t lo, hi;
          granule_span(dmis, len, G, k, &lo, &hi);
          const int64_t goff = doff - int64_t(dmis) + 16 * int64_t(k);
          if (lo == 0 && hi == 16) {
            for (int j = 0; j < R; ++j) __stcs(reinterpret_cast<uint4*>(dptr[j] + goff), v);
          } else {
            for (int j = 0; j < R; ++j) store_partial16(dptr[j] + goff, v, lo, hi);
          }
        } else {
          for (int j = 0; j < R; ++j) {
            const uint32_t dm = uint32_t(reinterpret_cast<uintptr_t>(dptr[j] + doff) & 15u);
            const uint32_t Gj = (dm + len + 15u) >> 4;
            if (k < Gj) put_granule(dptr[j], doff, dm, len, Gj, k, granule(stage, spos, dm, k));
          }
        }
      };
      if (nr == 1) {
        // one row (a piece of a run or of a long row): its offsets once per stage
        const int64_t doff = row_doff[s][0];
        const uint32_t spos = row_spos[s][0];
        const uint32_t dmis = uint32_t(reinterpret_cast<uintptr_t>(dptr[0] + doff) & 15u);
        const uint32_t G = (dmis + len + 15u) >> 4;
        const uint32_t kend = bulk || congruent ? G : gmax;
        for (uint32_t k = ct; k < kend; k += kConsumerThreads) item(0, k, doff, spos, dmis, G);
      } else {
        const FastDiv32 by_g(gmax);
        const uint32_t items = nr * gmax;
        for (uint32_t i = ct; i < items; i += kConsumerThreads) {
          const uint32_t r = by_g.div(i);
          const uint32_t k = i - r * gmax;
          const int64_t doff = row_doff[s][r];
          const uint32_t dmis = uint32_t(reinterpret_cast<uintptr_t>(dptr[0] + doff) & 15u);
          item(r, k, doff, row_spos[s][r], dmis, (dmis + len + 15u) >> 4);
        }
      }
      if (bulk) {
        // make the output stage visible to the bulk copies, then hand it over
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive(&out_full[o]);
      } else {
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
      }
      ++n;
    }
  } else if (bulk) {
    // ------------------------------------------------------------ store warp
    while (true) {
      const int s = int(n % kStages), o = int(n % kOutStages);
      if (!warp_wait(&out_full[o], (n / kOutStages) & 1u)) {
        if (lane == 0) atomicExch(status, kStatusConsumerWait);
        break;
      }
      const StageDesc c = desc[s];
      if (c.ti < 0) break;
      const uint32_t R = desc_R[s];
      const uint32_t nr = c.kind == 1 ? uint32_t(c.b - c.a) : 1u;
      const uint32_t len = desc_len[s];
      const uint32_t ost = Walker::out_stride(len);
      const unsigned char* out = out_mem + size_t(o) * kStageBytes;
      unsigned char* const* dptr = dst_ptr[s];
      for (uint32_t q = lane; q < nr * R; q += 32) {
        const uint32_t r = q / R, j = q - r * R;
        const int64_t doff = row_doff[s][r];
        const uint32_t dmis = uint32_t(reinterpret_cast<uintptr_t>(dptr[0] + doff) & 15u);
        const uint32_t G = (dmis + len + 15u) >> 4;
        const uint32_t kf = dmis != 0 ? 1u : 0u;                          // first whole granule
        const uint32_t ke = G - (((dmis + len) & 15u) != 0 ? 1u : 0u);  // one past the last
        if (ke > kf)
          bulk_store(dptr[j] + doff - int64_t(dmis) + 16 * int64_t(kf),
                     out + size_t(r) * ost + 16u * kf, 16u * (ke - kf));
      }
      bulk_commit();
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);  // row table and pointers read
      bulk_wait_read_all_but_newest();
      __syncwarp();
      if (lane == 0 && n >= 1) mbar_arrive(&out_free[(n - 1) % kOutStages]);
      ++n;
    }
    bulk_wait_all();
  }
  // every role is done (all waits above are bounded): count the CTA out
  __syncthreads();
  finish_queue(queue);
}

std::mutex g_mu;
struct DeviceInfo {
  bool ready = false;
  int blocks_per_sm[2] = {1, 1};  // [BULK]
};
constexpr int kMaxDevices = 256;
DeviceInfo g_info[kMaxDevices];

template <bool BULK>
cudaError_t prepare(int* blocks_per_sm) {
  const void* fn = reinterpret_cast<const void*>(realign_staged_kernel<BULK>);
  cudaError_t ce =
      cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, Config<BULK>::kDynSmem);
  if (ce != cudaSuccess) return ce;
  int nb = 0;
  ce = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, fn, Config<BULK>::kThreads,
                                                     Config<BULK>::kDynSmem);
  *blocks_per_sm = nb > 0 ? nb : 1;
  return ce;
}

}  // namespace

reshard_status_t launch_realign_staged(int num_sms, const KernelParams& kp, const Program& prog,
                                       void* stream) {
  unsigned int* status = nullptr;
  reshard_status_t st = device_status_word(&status);
  if (st != RESHARD_OK) return st;
  int dev = -1;
  cudaError_t ce = cudaGetDevice(&dev);
  if (ce != cudaSuccess)
    return fail(RESHARD_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(ce));
  if (dev < 0 || dev >= kMaxDevices) return fail(RESHARD_ERR_UNSUPPORTED, "device ordinal too large");
  const bool bulk = (kp.flags & kFlagDstCongruent) && (kp.flags & kFlagBulkStores);
  int bps = 1;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceInfo& d = g_info[dev];
    if (!d.ready) {
      ce = prepare<false>(&d.blocks_per_sm[0]);
      if (ce == cudaSuccess) ce = prepare<true>(&d.blocks_per_sm[1]);
      if (ce != cudaSuccess)
        return fail(RESHARD_ERR_CUDA, std::string("staged kernel setup: ") + cudaGetErrorString(ce));
      d.ready = true;
    }
    bps = d.blocks_per_sm[bulk ? 1 : 0];
  }
  const int64_t max_grid = int64_t(num_sms) * bps;
  const unsigned grid = unsigned(kp.total_units < max_grid ? kp.total_units : max_grid);
  KernelParams params = kp;
  QueueSlot slot;
  st = work_queue_acquire(stream, &slot);
  if (st != RESHARD_OK) return st;
  unsigned int* queue = slot.addr;
  // pieces of at least 16 KiB: tiny ones cost more in grabs and short chunks
  // than they gain in balance (measured on the small uneven-stress tensors)
  PieceSchedule sched = work_queue_schedule(kp.total_units, prog.tile_bytes, prog.write_bytes, grid,
                                            16 * 1024);
  void* args[] = {&params, &status, &queue, &sched};
  if (bulk)
    ce = cudaLaunchKernel(reinterpret_cast<const void*>(realign_staged_kernel<true>), dim3(grid),
                          dim3(Config<true>::kThreads), args, Config<true>::kDynSmem,
                          static_cast<cudaStream_t>(stream));
  else
    ce = cudaLaunchKernel(reinterpret_cast<const void*>(realign_staged_kernel<false>), dim3(grid),
                          dim3(Config<false>::kThreads), args, Config<false>::kDynSmem,
                          static_cast<cudaStream_t>(stream));
  st = work_queue_release(slot, stream, ce == cudaSuccess);
  if (ce != cudaSuccess)
    return fail(RESHARD_ERR_CUDA, std::string("kernel launch: ") + cudaGetErrorString(ce));
  return st;
}

}  // namespace rs
