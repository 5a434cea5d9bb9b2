// static_scratch.cu -- gather_broadcast_execute_static: the gather-and-broadcast
// baseline without any allocation, for callers that cannot call cudaMalloc.
//
// The full-tensor scratch and the gather/slice descriptor tables live in two
// file-scope static device arrays.  Host code never uses the arrays' names as
// addresses (in host code they are host-side stand-ins): the first call on a
// device looks the real device addresses up with cudaGetSymbolAddress, with
// that device current, and every call passes those addresses to the kernels.
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>
#include <string>

#include "internal.h"

namespace rs {
namespace {

static __device__ __align__(256) unsigned char g_static_scratch[RESHARD_STATIC_SCRATCH_BYTES];
static __device__ __align__(256) unsigned char g_static_tables[RESHARD_STATIC_TABLE_BYTES];

constexpr int kMaxDevices = 256;

struct StaticArrays {
  bool ready = false;
  unsigned char* scratch = nullptr;  // device address of g_static_scratch
  unsigned char* tables = nullptr;   // device address of g_static_tables
  int num_sms = 0;
};

std::mutex g_static_mu;
StaticArrays g_static[kMaxDevices];

// Once per device, with that device current: device addresses of the arrays.
reshard_status_t static_arrays(int dev, StaticArrays* out) {
  if (dev < 0 || dev >= kMaxDevices) return fail(RESHARD_ERR_UNSUPPORTED, "device ordinal too large");
  std::lock_guard<std::mutex> lk(g_static_mu);
  StaticArrays& a = g_static[dev];
  if (!a.ready) {
    void* p = nullptr;
    cudaError_t ce = cudaGetSymbolAddress(&p, g_static_scratch);
    if (ce != cudaSuccess)
      return fail(RESHARD_ERR_CUDA, std::string("cudaGetSymbolAddress(scratch): ") + cudaGetErrorString(ce));
    void* q = nullptr;
    ce = cudaGetSymbolAddress(&q, g_static_tables);
    if (ce != cudaSuccess)
      return fail(RESHARD_ERR_CUDA, std::string("cudaGetSymbolAddress(tables): ") + cudaGetErrorString(ce));
    int sms = 0;
    ce = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (ce != cudaSuccess)
      return fail(RESHARD_ERR_CUDA, std::string("device query: ") + cudaGetErrorString(ce));
    a.scratch = static_cast<unsigned char*>(p);
    a.tables = static_cast<unsigned char*>(q);
    a.num_sms = sms;
    a.ready = true;
  }
  *out = a;
  return RESHARD_OK;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Layout of one program's tables inside the static table array.
struct TableSlots {
  size_t tiles, prefix, goff, gbuf, end;
};

TableSlots place(const Program& p, size_t base) {
  TableSlots t;
  t.tiles = base;
  t.prefix = align256(t.tiles + p.tiles.size() * sizeof(reshard_tile_t));
  t.goff = align256(t.prefix + p.prefix.size() * sizeof(int64_t));
  t.gbuf = align256(t.goff + p.goff.size() * sizeof(uint32_t));
  t.end = align256(t.gbuf + p.gbuf.size() * sizeof(uint16_t));
  return t;
}

reshard_status_t copy_tables(const Program& p, const TableSlots& s, unsigned char* dtab,
                             cudaStream_t stream) {
  struct Piece {
    size_t off;
    const void* src;
    size_t bytes;
  } pieces[4] = {{s.tiles, p.tiles.data(), p.tiles.size() * sizeof(reshard_tile_t)},
                 {s.prefix, p.prefix.data(), p.prefix.size() * sizeof(int64_t)},
                 {s.goff, p.goff.data(), p.goff.size() * sizeof(uint32_t)},
                 {s.gbuf, p.gbuf.data(), p.gbuf.size() * sizeof(uint16_t)}};
  for (const Piece& pc : pieces) {
    if (pc.bytes == 0) continue;
    cudaError_t ce = cudaMemcpyAsync(dtab + pc.off, pc.src, pc.bytes, cudaMemcpyHostToDevice, stream);
    if (ce != cudaSuccess)
      return fail(RESHARD_ERR_CUDA, std::string("table copy: ") + cudaGetErrorString(ce));
  }
  return RESHARD_OK;
}

}  // namespace
}  // namespace rs

using rs::fail;

extern "C" reshard_status_t gather_broadcast_execute_static(reshard_plan_t plan,
                                                            const void* const* src_ptrs,
                                                            void* const* dst_ptrs, void* stream) {
  rs::TraceRange trace("gb.exec_static");
  if (!rs::plan_live(plan)) return fail(RESHARD_ERR_BAD_HANDLE, "invalid plan handle");
  const reshard_stats_t& st = plan->stats;
  if (uint64_t(st.global_bytes) > RESHARD_STATIC_SCRATCH_BYTES)
    return fail(RESHARD_ERR_UNSUPPORTED,
                "global tensor of " + std::to_string(st.global_bytes) +
                    " bytes exceeds the static scratch of " +
                    std::to_string(uint64_t(RESHARD_STATIC_SCRATCH_BYTES)) +
                    " bytes; use gather_broadcast_execute with a caller-owned scratch");
  const rs::Program& pg = plan->prog[RESHARD_PROGRAM_GATHER];
  const rs::Program& ps = plan->prog[RESHARD_PROGRAM_SLICE];
  const rs::TableSlots tg = rs::place(pg, 0);
  const rs::TableSlots ts = rs::place(ps, tg.end);
  if (ts.end > RESHARD_STATIC_TABLE_BYTES)
    return fail(RESHARD_ERR_UNSUPPORTED,
                "gather and slice tables of " + std::to_string(ts.end) +
                    " bytes exceed the static table array of " +
                    std::to_string(uint64_t(RESHARD_STATIC_TABLE_BYTES)) + " bytes");

  // buffer table [sources..., destinations..., scratch], with the same pointer
  // checks as every other execution (NULL for empty shards and for ranks an
  // excluded plan leaves out; source aliases of in-place plans); the scratch
  // slot is filled in below once the static array's address is known
  unsigned char* bufs[RESHARD_MAX_EXEC_BUFFERS];
  reshard_status_t rc =
      rs::buffer_table(plan, src_ptrs, dst_ptrs, nullptr, bufs, RESHARD_MAX_EXEC_BUFFERS);
  if (rc != RESHARD_OK) return rc;
  const int64_t M = plan->src.nranks, N = plan->dst.nranks;

  int dev = -1;
  cudaError_t ce = cudaGetDevice(&dev);
  if (ce != cudaSuccess)
    return fail(RESHARD_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(ce));
  rs::StaticArrays arr;
  rc = rs::static_arrays(dev, &arr);
  if (rc != RESHARD_OK) return rc;
  bufs[M + N] = arr.scratch;
  const int nbufs = int(M + N + 1);
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  rc = rs::copy_tables(pg, tg, arr.tables, s);
  if (rc == RESHARD_OK) rc = rs::copy_tables(ps, ts, arr.tables, s);
  if (rc != RESHARD_OK) return rc;
  unsigned char* t = arr.tables;
  rc = rs::launch_program_tables(pg, reinterpret_cast<const reshard_tile_t*>(t + tg.tiles),
                                 reinterpret_cast<const int64_t*>(t + tg.prefix),
                                 reinterpret_cast<const uint32_t*>(t + tg.goff),
                                 reinterpret_cast<const uint16_t*>(t + tg.gbuf), arr.num_sms, bufs,
                                 nbufs, stream);
  if (rc != RESHARD_OK) return rc;
  return rs::launch_program_tables(ps, reinterpret_cast<const reshard_tile_t*>(t + ts.tiles),
                                   reinterpret_cast<const int64_t*>(t + ts.prefix),
                                   reinterpret_cast<const uint32_t*>(t + ts.goff),
                                   reinterpret_cast<const uint16_t*>(t + ts.gbuf), arr.num_sms,
                                   bufs, nbufs, stream);
}
