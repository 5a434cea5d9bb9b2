// bulk_fanout.cu -- TMA-staged read-once fan-out (sm_103a), and the device
// status word shared by the library's kernels.
//
// Used for fan-out programs in which every tile offset, stride, row length and
// buffer address is a multiple of 16 bytes.  Each CTA runs a two-warp pipeline
// over its equal share of the program's work units (the same partition as the
// vector kernel in kernels.cu):
//   warp 0 (producer) copies the next chunk of source bytes -- a piece of a
//     contiguous run, a few whole rows, or a piece of a long row -- into a
//     ring of shared-memory stages with cp.async.bulk; completion is counted in
//     bytes on the stage's "full" mbarrier;
//   warp 1 (consumer) waits for the stage and writes it to every destination
//     replica of the tile with cp.async.bulk stores (rows that are contiguous
//     in the destination go out as one store per replica), commits them as a
//     bulk group and, once all but the newest group have been read out of
//     shared memory, releases the previous stage on its "empty" mbarrier.
// The source region crosses HBM once and is written R times by the TMA
// engine, without passing through registers.  No multicast is used.
//
// Every mbarrier wait is bounded.  A wait that runs out records a code in the
// device status word, waits (boundedly) for the CTA's own bulk copies and
// returns, so the context stays usable; reshard_device_status() reads it.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>
#include <string>

#include "internal.h"

namespace rs {
namespace {

constexpr int kStages = 2;
constexpr uint32_t kStageBytes = 32 * 1024;
constexpr int kStagedThreads = 64;
// try_wait polls before a wait is declared lost (a poll may suspend the thread
// for a short, hardware-defined time: this is of the order of a second).
constexpr uint32_t kWaitPolls = 1u << 22;

enum : unsigned int {
  kStatusProducerWait = 1,  // producer gave up waiting for a free stage
  kStatusConsumerWait = 2,  // consumer gave up waiting for a loaded stage
  kStatusSelfTest = 3       // the self-test's deliberately unanswered wait ran out
};

__device__ unsigned int g_device_status;

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

// One chunk: at most kStageBytes of one tile.
struct Chunk {
  int ti;
  uint32_t kind;   // 0: piece [a, b) of a run; 1: whole rows [a, b); 2: bytes [b, b+bytes) of row a
  int64_t a, b;
  uint32_t bytes;
};

// Walks the chunks of this CTA's unit range; the producer and the consumer each
// run their own copy and see the same sequence.
struct ChunkWalker {
  const KernelParams* p;
  int64_t u0, u1;
  int ti;
  int64_t pos, end;
  uint32_t kind, per;  // per: rows per chunk (kind 1) or pieces per row (kind 2)
  reshard_tile_t t;
  bool live;

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
    const int64_t upr = t.row_bytes >= kUnitBytes ? 1 : kUnitBytes / t.row_bytes;
    const int64_t rows = int64_t(t.nrows) * t.nplanes;
    const int64_t r0 = a * upr, r1 = min(b * upr, rows);
    if (t.row_bytes <= kStageBytes) {
      kind = 1;
      per = kStageBytes / t.row_bytes;
      pos = r0;
      end = r1;
    } else {
      kind = 2;
      per = (t.row_bytes + kStageBytes - 1) / kStageBytes;
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
      const int64_t e = min(end, pos + int64_t(kStageBytes));
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
      const int64_t b0 = piece * kStageBytes;
      const int64_t b1 = min(int64_t(t.row_bytes), b0 + int64_t(kStageBytes));
      c->a = row;
      c->b = b0;
      c->bytes = uint32_t(b1 - b0);
      pos += 1;
    }
    return true;
  }
};

__device__ __forceinline__ int64_t src_row(const reshard_tile_t& t, int64_t r) {
  const int64_t pl = r / t.nrows, q = r - pl * t.nrows;
  return t.src_off + pl * t.src_plane_stride + q * t.src_row_stride;
}
__device__ __forceinline__ int64_t dst_row(const reshard_tile_t& t, int64_t r) {
  const int64_t pl = r / t.nrows, q = r - pl * t.nrows;
  return t.dst_off + pl * t.dst_plane_stride + q * t.dst_row_stride;
}

__global__ void __launch_bounds__(kStagedThreads)
    fanout_staged_kernel(const __grid_constant__ KernelParams p, unsigned int* status) {
  extern __shared__ __align__(1024) unsigned char stage_mem[];
  __shared__ __align__(8) uint64_t full[kStages], empty[kStages];
  __shared__ unsigned char* dst_base[kMaxGroup];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  ChunkWalker w;
  w.start(&p);
  Chunk c;
  uint32_t n = 0;
  if (warp == 0) {
    // producer: source -> stage (n % kStages)
    while (w.next(&c)) {
      const int s = int(n % kStages);
      if (n >= uint32_t(kStages) &&
          !mbar_wait(&empty[s], ((n / kStages) - 1) & 1u, kWaitPolls)) {
        if (lane == 0) atomicExch(status, kStatusProducerWait);
        return;  // nothing of ours is in flight that this stage still needs
      }
      unsigned char* buf = stage_mem + size_t(s) * kStageBytes;
      const reshard_tile_t& t = w.t;
      const unsigned char* src = p.bufs[t.src_buf];
      if (lane == 0) mbar_arrive_expect(&full[s], c.bytes);
      __syncwarp();
      if (c.kind == 0) {
        if (lane == 0) bulk_load(buf, src + t.src_off + c.a, c.bytes, &full[s]);
      } else if (c.kind == 1) {
        for (int64_t r = c.a + lane; r < c.b; r += 32)
          bulk_load(buf + (r - c.a) * t.row_bytes, src + src_row(t, r), t.row_bytes, &full[s]);
      } else {
        if (lane == 0) bulk_load(buf, src + src_row(t, c.a) + c.b, c.bytes, &full[s]);
      }
      ++n;
    }
  } else {
    // consumer: stage -> every destination replica
    int cur_tile = -1, R = 0;
    while (w.next(&c)) {
      const int s = int(n % kStages);
      const reshard_tile_t& t = w.t;
      if (c.ti != cur_tile) {
        const uint32_t g0 = p.goff[t.dst_group];
        R = int(p.goff[t.dst_group + 1] - g0);
        for (int i = lane; i < R; i += 32) dst_base[i] = p.bufs[p.gbuf[g0 + i]];
        __syncwarp();
        cur_tile = c.ti;
      }
      if (!mbar_wait(&full[s], (n / kStages) & 1u, kWaitPolls)) {
        if (lane == 0) atomicExch(status, kStatusConsumerWait);
        break;
      }
      const unsigned char* buf = stage_mem + size_t(s) * kStageBytes;
      if (c.kind == 0) {
        for (int r = lane; r < R; r += 32) bulk_store(dst_base[r] + t.dst_off + c.a, buf, c.bytes);
      } else if (c.kind == 1) {
        if (t.nplanes == 1 && t.dst_row_stride == int64_t(t.row_bytes)) {
          for (int r = lane; r < R; r += 32)
            bulk_store(dst_base[r] + dst_row(t, c.a), buf, c.bytes);
        } else {
          const int64_t nr = c.b - c.a;
          for (int64_t k = lane; k < nr * R; k += 32) {
            const int64_t row = k / R, r = k - row * R;
            bulk_store(dst_base[r] + dst_row(t, c.a + row), buf + row * t.row_bytes, t.row_bytes);
          }
        }
      } else {
        for (int r = lane; r < R; r += 32)
          bulk_store(dst_base[r] + dst_row(t, c.a) + c.b, buf, c.bytes);
      }
      bulk_commit();
      bulk_wait_read_all_but_newest();
      __syncwarp();
      if (lane == 0 && n >= 1) mbar_arrive(&empty[(n - 1) % kStages]);
      ++n;
    }
    bulk_wait_all();
  }
}

// A wait that nothing will ever answer: exercises the bounded-wait path.
__global__ void selftest_wait_kernel(unsigned int* status, uint32_t polls) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (threadIdx.x == 0 && !mbar_wait(&bar, 0, polls)) atomicExch(status, kStatusSelfTest);
}

constexpr int kMaxDevices = 256;
struct DeviceState {
  bool ready = false;
  unsigned int* status = nullptr;  // device address of g_device_status
  int blocks_per_sm = 0;
};
std::mutex g_dev_mu;
DeviceState g_dev[kMaxDevices];

reshard_status_t device_state(DeviceState* out) {
  int dev = -1;
  cudaError_t ce = cudaGetDevice(&dev);
  if (ce != cudaSuccess)
    return fail(RESHARD_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(ce));
  if (dev < 0 || dev >= kMaxDevices) return fail(RESHARD_ERR_UNSUPPORTED, "device ordinal too large");
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceState& d = g_dev[dev];
  if (!d.ready) {
    void* addr = nullptr;
    ce = cudaGetSymbolAddress(&addr, g_device_status);
    if (ce != cudaSuccess)
      return fail(RESHARD_ERR_CUDA, std::string("cudaGetSymbolAddress: ") + cudaGetErrorString(ce));
    const int smem = kStages * int(kStageBytes);
    ce = cudaFuncSetAttribute(reinterpret_cast<const void*>(fanout_staged_kernel),
                              cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (ce != cudaSuccess)
      return fail(RESHARD_ERR_CUDA, std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(ce));
    int n = 0;
    ce = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        &n, reinterpret_cast<const void*>(fanout_staged_kernel), kStagedThreads, smem);
    if (ce != cudaSuccess)
      return fail(RESHARD_ERR_CUDA, std::string("occupancy query: ") + cudaGetErrorString(ce));
    d.status = static_cast<unsigned int*>(addr);
    d.blocks_per_sm = n > 0 ? n : 1;
    d.ready = true;
  }
  *out = d;
  return RESHARD_OK;
}

}  // namespace

reshard_status_t launch_fanout_staged(const reshard_plan_s* plan, const KernelParams& kp,
                                      void* stream) {
  DeviceState d;
  reshard_status_t st = device_state(&d);
  if (st != RESHARD_OK) return st;
  const int64_t max_grid = int64_t(plan->num_sms) * d.blocks_per_sm;
  const unsigned grid = unsigned(kp.total_units < max_grid ? kp.total_units : max_grid);
  KernelParams params = kp;
  unsigned int* status = d.status;
  void* args[] = {&params, &status};
  cudaError_t ce = cudaLaunchKernel(reinterpret_cast<const void*>(fanout_staged_kernel),
                                    dim3(grid), dim3(kStagedThreads), args,
                                    kStages * kStageBytes, static_cast<cudaStream_t>(stream));
  if (ce != cudaSuccess)
    return fail(RESHARD_ERR_CUDA, std::string("kernel launch: ") + cudaGetErrorString(ce));
  return RESHARD_OK;
}

}  // namespace rs

using rs::fail;

extern "C" {

reshard_status_t reshard_device_status(int32_t clear, uint32_t* status) {
  if (!status) return fail(RESHARD_ERR_INVALID_ARG, "status is NULL");
  rs::DeviceState d;
  reshard_status_t st = rs::device_state(&d);
  if (st != RESHARD_OK) return st;
  unsigned int v = 0;
  cudaError_t ce = cudaMemcpy(&v, d.status, sizeof(v), cudaMemcpyDeviceToHost);
  if (ce != cudaSuccess)
    return fail(RESHARD_ERR_CUDA, std::string("status read: ") + cudaGetErrorString(ce));
  if (clear) {
    ce = cudaMemset(d.status, 0, sizeof(unsigned int));
    if (ce != cudaSuccess)
      return fail(RESHARD_ERR_CUDA, std::string("status clear: ") + cudaGetErrorString(ce));
  }
  *status = v;
  return RESHARD_OK;
}

reshard_status_t reshard_selftest_wait_timeout(uint32_t polls, void* stream) {
  rs::DeviceState d;
  reshard_status_t st = rs::device_state(&d);
  if (st != RESHARD_OK) return st;
  if (polls == 0 || polls > (1u << 20)) return fail(RESHARD_ERR_INVALID_ARG, "polls must be 1..2^20");
  unsigned int* status = d.status;
  void* args[] = {&status, &polls};
  cudaError_t ce = cudaLaunchKernel(reinterpret_cast<const void*>(rs::selftest_wait_kernel), dim3(1),
                                    dim3(32), args, 0, static_cast<cudaStream_t>(stream));
  if (ce != cudaSuccess)
    return fail(RESHARD_ERR_CUDA, std::string("kernel launch: ") + cudaGetErrorString(ce));
  return RESHARD_OK;
}

}  // extern "C"
