// bulk_fanout.cu -- TMA-staged read-once fan-out (sm_103a), and the device
// status word shared by the library's kernels.
//
// Used for fan-out programs in which every tile offset, stride, row length and
// buffer address is a multiple of 16 bytes.  Each CTA runs a two-warp pipeline
// over pieces of consecutive work units that it takes from a per-launch work
// queue as it goes, so that CTAs on faster SMs take more pieces and all finish
// together (a static equal split left the slowest SMs 15-25% behind):
//   warp 0 (producer) takes pieces and copies their chunks of source bytes --
//     a piece of a contiguous run, a few whole rows, or a piece of a long row --
//     into a ring of shared-memory stages with cp.async.bulk, with a descriptor
//     of the chunk beside each stage; completion is counted in bytes on the
//     stage's "full" mbarrier; a descriptor with no tile ends the CTA's work;
//   warp 1 (consumer) waits for the stage and writes it to every destination
//     replica of the tile with cp.async.bulk stores (rows that are contiguous
//     in the destination go out as one store per replica), commits them as a
//     bulk group and, once all but the newest group have been read out of
//     shared memory, releases the previous stage on its "empty" mbarrier.
// The source region crosses HBM once and is written R times by the TMA
// engine, without passing through registers.  No multicast is used.
//
// Every mbarrier wait is bounded.  A wait that runs out records a code in the
// device status word, waits (boundedly) for the CTA's own bulk copies -- the
// loads into its stages as well as its stores -- and returns, so the context
// stays usable; reshard_device_status() reads it.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <map>
#include <mutex>
#include <string>
#include <thread>
#include <utility>

#include "internal.h"
#include "staging.cuh"

namespace rs {
namespace {

using namespace staging;

constexpr int kStages = 2;
constexpr uint32_t kStageBytes = 32 * 1024;
constexpr int kStagedThreads = 64;

__device__ unsigned int g_device_status;

// Work queue: pieces of consecutive work units are handed to CTAs in order as
// they ask, so CTAs that run fast take more pieces and all finish
// together.  Every launch takes its own slot {next piece, CTAs finished}; the
// last CTA of the launch puts the slot back to zero.
// Slots [0, kStreamSlots) belong to streams, one each at a time (a slot passes to
// another stream once its last launch has finished, see SlotTable); the rest go
// to launches captured into CUDA graphs, one each, never handed out again (a
// graph may be replayed on any stream, beside the eager launches of the stream
// it came from).
constexpr int kQueueSlots = 4096;
constexpr int kStreamSlots = 1024;
__device__ unsigned int g_queue[kQueueSlots][2];
// Units per piece: about kPieceBytes of the program's bytes, and few enough
// that every CTA can get about kPiecesPerCta pieces (small programs still use
// the whole grid).  Measured: 32 KiB pieces beat 8-unit and 64 KiB ones over
// the workloads taken together.  The last kTailRounds pieces per CTA are cut
// kTailDiv times smaller: a CTA holds up to two pieces (the one it works on
// and the one it has already asked for), so big last pieces leave some SMs
// busy for two piece-times after the others ran out of work.  A tail piece
// still moves at least kTailPieceTraffic bytes (read plus written): shorter
// ones were measured slower on one-to-one copies.
constexpr int64_t kPieceBytes = 32 * 1024;
constexpr int64_t kPiecesPerCta = 8;
constexpr int64_t kTailRounds = 2;
constexpr int64_t kTailDiv = 4;
constexpr int64_t kTailPieceTraffic = 40 * 1024;

__global__ void __launch_bounds__(kStagedThreads)
    fanout_staged_kernel(const __grid_constant__ KernelParams p, unsigned int* status,
                         unsigned int* queue, const PieceSchedule sched) {
  extern __shared__ __align__(1024) unsigned char stage_mem[];
  __shared__ __align__(8) uint64_t full[kStages], empty[kStages];
  __shared__ StageDesc desc[kStages];
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

  uint32_t n = 0;
  if (warp == 0) {
    // producer: pieces from the queue -> chunks -> stage (n % kStages)
    ChunkWalker<kStageBytes, 0> w;
    Chunk c;
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
        if (n >= uint32_t(kStages) &&
            !mbar_wait(&empty[s], ((n / kStages) - 1) & 1u, kWaitPolls)) {
          if (lane == 0) atomicExch(status, kStatusProducerWait);
          ok = false;
          break;
        }
        unsigned char* buf = stage_mem + size_t(s) * kStageBytes;
        const reshard_tile_t& t = w.t;
        const unsigned char* src = p.bufs[t.src_buf];
        if (lane == 0) {
          desc[s] = StageDesc{c.ti, c.kind, c.bytes, c.a, c.b};
          mbar_arrive_expect(&full[s], c.bytes);
        }
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
      piece = next_piece;
    }
    // end marker: a stage whose descriptor says "no more chunks", with no bytes
    if (ok) {
      const int s = int(n % kStages);
      if (n >= uint32_t(kStages) && !mbar_wait(&empty[s], ((n / kStages) - 1) & 1u, kWaitPolls)) {
        if (lane == 0) atomicExch(status, kStatusProducerWait);
      } else {
        if (lane == 0) {
          desc[s].ti = -1;
          mbar_arrive(&full[s]);
        }
        ++n;
      }
    }
    // wait (boundedly) for the copies still landing in the stages: after a wait
    // ran out, the consumer may have stopped before reading them, and the CTA
    // must not exit while bulk copies still write its shared memory.  Each of
    // the last kStages stages is waited on at the phase of its latest use (on
    // the normal path those phases have completed and the waits return at once).
    const uint32_t issued = n;
    for (uint32_t m = issued > uint32_t(kStages) ? issued - kStages : 0u; m < issued; ++m)
      mbar_wait(&full[m % kStages], (m / kStages) & 1u, kWaitPolls);
  } else {
    // consumer: stage -> every destination replica
    int cur_tile = -1, R = 0;
    reshard_tile_t t = {};
    while (true) {
      const int s = int(n % kStages);
      if (!mbar_wait(&full[s], (n / kStages) & 1u, kWaitPolls)) {
        if (lane == 0) atomicExch(status, kStatusConsumerWait);
        break;
      }
      const StageDesc c = desc[s];
      if (c.ti < 0) break;
      if (c.ti != cur_tile) {
        t = p.tiles[c.ti];
        const uint32_t g0 = p.goff[t.dst_group];
        R = int(p.goff[t.dst_group + 1] - g0);
        for (int i = lane; i < R; i += 32) dst_base[i] = p.bufs[p.gbuf[g0 + i]];
        __syncwarp();
        cur_tile = c.ti;
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
  // both roles are done (every wait above is bounded): count the CTA out, and
  // the last one puts the launch's queue slot back to zero
  __syncthreads();
  finish_queue(queue);
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
  unsigned int* queue = nullptr;   // device address of g_queue
  int blocks_per_sm = 0;
};
std::mutex g_dev_mu;
// Per device, the stream slots: which stream holds each one, an event recorded
// on that stream after the slot's latest launch, and whether a launch is between
// acquire and release.  A slot changes hands only when its event reports that
// the slot's last launch has finished (the launch's last CTA has put it back to
// zero), or, when no slot is idle, after the new stream has been made to wait
// for that event.  Streams are told apart by their unique ids (a handle can be
// reused after a stream is destroyed); the per-thread default stream also by
// thread.
using StreamKey = std::pair<unsigned long long, std::thread::id>;
struct StreamSlot {
  StreamKey key{};
  bool held = false;         // some stream holds the slot
  bool busy = false;         // acquired, launch not yet released
  cudaEvent_t done = nullptr;  // recorded after the slot's latest launch
  uint64_t last_use = 0;
};
struct SlotTable {
  std::map<StreamKey, uint32_t> by_stream;
  StreamSlot slot[kStreamSlots];
  uint32_t next_stream = 0;
  uint32_t next_captured = kStreamSlots;
  uint64_t clock = 0;
};
std::mutex g_slot_mu;
DeviceState g_dev[kMaxDevices];
SlotTable g_slots[kMaxDevices];

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
    void* qaddr = nullptr;
    ce = cudaGetSymbolAddress(&qaddr, g_queue);
    if (ce != cudaSuccess)
      return fail(RESHARD_ERR_CUDA, std::string("cudaGetSymbolAddress: ") + cudaGetErrorString(ce));
    d.queue = static_cast<unsigned int*>(qaddr);
    d.status = static_cast<unsigned int*>(addr);
    d.blocks_per_sm = n > 0 ? n : 1;
    d.ready = true;
  }
  *out = d;
  return RESHARD_OK;
}

}  // namespace

reshard_status_t work_queue_acquire(void* stream, QueueSlot* q) {
  DeviceState d;
  reshard_status_t st = device_state(&d);
  if (st != RESHARD_OK) return st;
  int dev = -1;
  cudaError_t ce = cudaGetDevice(&dev);
  if (ce != cudaSuccess)
    return fail(RESHARD_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(ce));
  cudaStream_t cs_stream = static_cast<cudaStream_t>(stream);
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  ce = cudaStreamIsCapturing(cs_stream, &cs);
  if (ce != cudaSuccess)
    return fail(RESHARD_ERR_CUDA, std::string("cudaStreamIsCapturing: ") + cudaGetErrorString(ce));
  std::lock_guard<std::mutex> lk(g_slot_mu);
  SlotTable& t = g_slots[dev];
  q->dev = dev;
  if (cs != cudaStreamCaptureStatusNone) {
    if (t.next_captured >= uint32_t(kQueueSlots))
      return fail(RESHARD_ERR_UNSUPPORTED, "more than " + std::to_string(kQueueSlots - kStreamSlots) +
                                               " work-queue launches captured into CUDA graphs "
                                               "on this device");
    q->idx = -1;  // captured: a slot of its own for good, no event
    q->addr = d.queue + 2 * t.next_captured++;
    return RESHARD_OK;
  }
  unsigned long long id = 0;
  if (cudaStreamGetId(cs_stream, &id) != cudaSuccess) {
    cudaGetLastError();  // clear the failed query from the library's runtime
    id = static_cast<unsigned long long>(reinterpret_cast<uintptr_t>(stream));
  }
  const StreamKey key(id, cs_stream == cudaStreamPerThread ? std::this_thread::get_id()
                                                           : std::thread::id());
  auto it = t.by_stream.find(key);
  uint32_t idx = 0;
  if (it != t.by_stream.end()) {
    idx = it->second;  // this stream's own slot: its launches run in turn
  } else {
    bool wait_for_previous = false;
    if (t.next_stream < uint32_t(kStreamSlots)) {
      idx = t.next_stream++;
    } else {
      // every slot has been used: take an idle one (its last launch has finished),
      // the least recently used first; if none is idle, the least recently used
      // one, after which the new stream waits for its last launch
      uint32_t order[kStreamSlots];
      uint32_t nfree = 0;
      for (uint32_t i = 0; i < uint32_t(kStreamSlots); ++i)
        if (!t.slot[i].busy) order[nfree++] = i;
      std::sort(order, order + nfree, [&t](uint32_t a, uint32_t b) {
        return t.slot[a].last_use < t.slot[b].last_use;
      });
      int64_t idle = -1;
      bool pending = false;
      for (uint32_t k = 0; k < nfree && idle < 0; ++k) {
        const StreamSlot& sl = t.slot[order[k]];
        const cudaError_t q = sl.done ? cudaEventQuery(sl.done) : cudaSuccess;
        if (q == cudaSuccess) idle = order[k];
        else pending = true;
      }
      // the library's own runtime records cudaErrorNotReady of a pending event
      // as its last error: clear it, it is not an error
      if (pending) cudaGetLastError();
      if (idle >= 0) {
        idx = uint32_t(idle);
      } else if (nfree > 0) {
        idx = order[0];
        wait_for_previous = true;
      } else {
        return fail(RESHARD_ERR_UNSUPPORTED,
                    "all " + std::to_string(kStreamSlots) +
                        " work-queue slots of this device are between acquire and launch");
      }
      if (t.slot[idx].held) t.by_stream.erase(t.slot[idx].key);
    }
    StreamSlot& sl = t.slot[idx];
    if (wait_for_previous && sl.done) {
      ce = cudaStreamWaitEvent(cs_stream, sl.done, 0);
      if (ce != cudaSuccess)
        return fail(RESHARD_ERR_CUDA, std::string("cudaStreamWaitEvent: ") + cudaGetErrorString(ce));
    }
    sl.key = key;
    sl.held = true;
    t.by_stream.emplace(key, idx);
  }
  t.slot[idx].busy = true;
  q->idx = int(idx);
  q->addr = d.queue + 2 * idx;
  return RESHARD_OK;
}

reshard_status_t work_queue_release(const QueueSlot& q, void* stream, bool launched) {
  if (q.idx < 0) return RESHARD_OK;
  std::lock_guard<std::mutex> lk(g_slot_mu);
  StreamSlot& sl = g_slots[q.dev].slot[q.idx];
  sl.busy = false;
  if (!launched) return RESHARD_OK;
  sl.last_use = ++g_slots[q.dev].clock;
  cudaError_t ce = cudaSuccess;
  if (!sl.done) ce = cudaEventCreateWithFlags(&sl.done, cudaEventDisableTiming);
  if (ce == cudaSuccess) ce = cudaEventRecord(sl.done, static_cast<cudaStream_t>(stream));
  if (ce != cudaSuccess) {
    // without a record the slot can no longer be shown idle: keep it with its stream
    sl.busy = true;
    return fail(RESHARD_ERR_CUDA, std::string("work-queue event: ") + cudaGetErrorString(ce));
  }
  return RESHARD_OK;
}

PieceSchedule work_queue_schedule(int64_t total_units, int64_t tile_bytes, int64_t write_bytes,
                                  int64_t grid, int64_t min_piece_bytes) {
  const int64_t units = total_units > 0 ? total_units : 1;
  const int64_t cta = grid > 0 ? grid : 1;
  const int64_t unit_bytes = tile_bytes / units > 0 ? tile_bytes / units : 1;
  const int64_t most = (kPieceBytes + unit_bytes - 1) / unit_bytes;
  // no smaller than min_piece_bytes while every CTA still gets a piece
  const int64_t least = std::min((min_piece_bytes + unit_bytes - 1) / unit_bytes,
                                 std::max<int64_t>(1, units / cta));
  const int64_t piece_units = std::max(units / (cta * kPiecesPerCta), least);
  PieceSchedule s;
  s.total = total_units > 0 ? total_units : 0;
  s.big = std::max<int64_t>(1, std::min(piece_units, most));
  const int64_t unit_traffic = std::max<int64_t>(1, (tile_bytes + write_bytes) / units);
  s.small = std::max({std::min(s.big, least), s.big / kTailDiv,
                      (kTailPieceTraffic + unit_traffic - 1) / unit_traffic, int64_t(1)});
  s.small = std::min(s.small, s.big);
  const int64_t tail = kTailRounds * cta * s.big;
  s.split = s.total > tail ? (s.total - tail) / s.big * s.big : 0;
  return s;
}

reshard_status_t device_status_word(unsigned int** status) {
  DeviceState d;
  reshard_status_t st = device_state(&d);
  if (st != RESHARD_OK) return st;
  *status = d.status;
  return RESHARD_OK;
}

reshard_status_t launch_fanout_staged(const reshard_plan_s* plan, const KernelParams& kp,
                                      const Program& prog, void* stream) {
  DeviceState d;
  reshard_status_t st = device_state(&d);
  if (st != RESHARD_OK) return st;
  const int64_t max_grid = int64_t(plan->num_sms) * d.blocks_per_sm;
  const unsigned grid = unsigned(kp.total_units < max_grid ? kp.total_units : max_grid);
  KernelParams params = kp;
  unsigned int* status = d.status;
  QueueSlot slot;
  st = work_queue_acquire(stream, &slot);
  if (st != RESHARD_OK) return st;
  unsigned int* queue = slot.addr;
  PieceSchedule sched = work_queue_schedule(kp.total_units, prog.tile_bytes, prog.write_bytes,
                                            grid, 0);
  void* args[] = {&params, &status, &queue, &sched};
  cudaError_t ce = cudaLaunchKernel(reinterpret_cast<const void*>(fanout_staged_kernel),
                                    dim3(grid), dim3(kStagedThreads), args,
                                    kStages * kStageBytes, static_cast<cudaStream_t>(stream));
  st = work_queue_release(slot, stream, ce == cudaSuccess);
  if (ce != cudaSuccess)
    return fail(RESHARD_ERR_CUDA, std::string("kernel launch: ") + cudaGetErrorString(ce));
  return st;
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
