// internal.h -- shared between the host planner (planner.cpp) and the CUDA
// kernels (kernels.cu) of libreshard.so.  Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <mutex>
#include <string>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "reshard.h"

namespace rs {

// A named NVTX range over a host call (plan creation, execution enqueue), so
// timelines show where the library's time goes; free when no tool is attached.
struct TraceRange {
  explicit TraceRange(const char* name) { nvtxRangePushA(name); }
  ~TraceRange() { nvtxRangePop(); }
  TraceRange(const TraceRange&) = delete;
  TraceRange& operator=(const TraceRange&) = delete;
};

// A multi-row tile whose rows are longer than this is split into one
// single-row ("run") tile per row, so that work units stay small.
constexpr int64_t kRunSplitBytes = 64 * 1024;
// Work-unit size of a single-row tile, and the row budget of a multi-row unit.
constexpr int64_t kUnitBytes = 4096;
// Largest single-row tile (longer runs are cut into several tiles).
constexpr int64_t kMaxRunBytes = int64_t(1) << 30;
// A multi-row fan-out tile that fills a column band of wider destination rows
// and goes to at least kGatherBlockFanout replicas is cut into blocks of about
// kGatherBlockBytes of rows, so that after the sort by destination offset the
// blocks of neighbouring bands interleave and each CTA writes whole stretches
// of destination rows to every replica (measured: it pays where writes
// dominate, and costs more tiles and smaller chunks elsewhere).  The blocks are
// small enough that the two pieces meeting in a 32-byte destination sector are
// written before L2 evicts the first half (a 15-replica fan-out of 628-byte
// rows: 0.615 / 0.569 / 0.549 / 0.579 ms at 32 / 16 / 8 / 4 KiB blocks).
constexpr int64_t kGatherBlockBytes = 8 * 1024;
constexpr int64_t kGatherBlockFanout = 8;
// Largest destination group one tile fans out to (larger groups are split).
constexpr int kMaxGroup = 256;

// Programs a plan holds: the four of reshard_program_t and the replicate step.
constexpr int kNumPrograms = 5;
// A destination class with at least this many replicas whose copies would go
// through the register realigning kernel (tiles off the 16-byte grid, mostly in
// rows of 512 bytes to 8 KiB) is assembled in one replica and then copied to the
// others as one aligned run (RESHARD_PROGRAM_REPLICATE).  Measured on GB300, a
// 138 MB fp32 gather of 56 pieces of 628 bytes into 15 replicas: 0.553 -> 0.386 ms;
// a 62 MB bf16 gather of 17 pieces of 770 bytes into 6 replicas: 0.119 -> 0.108 ms.
constexpr int64_t kAssembleFanout = 6;

// Rows shorter than this count as narrow (the element kernel keeps fewer
// loads in flight for programs made mostly of them).
constexpr int64_t kNarrowRow = 32;

// Fixed work of one row (offsets, partial first and last words, a row-table
// entry), counted in bytes of streaming when rows are grouped into units.
constexpr int64_t kRowCostBytes = 256;

#ifdef __CUDACC__
#define RS_HOST_DEVICE __host__ __device__
#else
#define RS_HOST_DEVICE
#endif

// Rows per work unit of a multi-row tile: rows whose bytes plus fixed work
// come to about kUnitBytes (at least one).
RS_HOST_DEVICE inline uint32_t rows_per_unit(uint32_t row_bytes) {
  const int64_t cost = int64_t(row_bytes) + kRowCostBytes;
  return cost >= kUnitBytes ? 1u : uint32_t(kUnitBytes / cost);
}

// Work units of a tile (must match the kernels' reading of a tile).
inline int64_t tile_units(const reshard_tile_t& t) {
  if (t.nrows == 1 && t.nplanes == 1) return (int64_t(t.row_bytes) + kUnitBytes - 1) / kUnitBytes;
  const int64_t rows = int64_t(t.nrows) * int64_t(t.nplanes);
  const int64_t upr = rows_per_unit(t.row_bytes);
  return (rows + upr - 1) / upr;
}

// Parameter block of the copy kernels: the program's device tables and the
// per-call buffer table (sources, destinations, scratch), passed by value.
struct KernelParams {
  const reshard_tile_t* tiles;
  const int64_t* prefix;
  const uint32_t* goff;
  const uint16_t* gbuf;
  int64_t total_units;
  int32_t ntiles;
  int32_t nbufs;
  uint32_t flags;  // kFlag* bits below
  uint32_t pad;
  unsigned char* bufs[RESHARD_MAX_EXEC_BUFFERS];
};
constexpr uint32_t kFlagDstCongruent = 1u;
// The realigning staged kernel writes whole granules with bulk copies from an
// output stage (only together with kFlagDstCongruent).
constexpr uint32_t kFlagBulkStores = 2u;

struct Box {
  int64_t off[RESHARD_MAX_TENSOR_NDIM];
  int64_t shp[RESHARD_MAX_TENSOR_NDIM];
};

struct Layout {
  int32_t mesh_ndim = 0;
  int64_t mesh[RESHARD_MAX_MESH_NDIM] = {};
  reshard_placement_t pl[RESHARD_MAX_MESH_NDIM] = {};
  int64_t nranks = 0;
  std::vector<Box> box;  // per flat rank
};

// One copy program: tiles in execution order, the units prefix, and the
// destination groups (lists of buffer indices).
struct Program {
  std::vector<reshard_tile_t> tiles;
  std::vector<int64_t> prefix;     // ntiles + 1
  std::vector<uint32_t> goff;      // ngroups + 1
  std::vector<uint16_t> gbuf;      // buffer indices
  // device copies (inside the plan's single device allocation)
  const reshard_tile_t* d_tiles = nullptr;
  const int64_t* d_prefix = nullptr;
  const uint32_t* d_goff = nullptr;
  const uint16_t* d_gbuf = nullptr;
  // OR of every tile's offsets, strides and row length (alignment class)
  uint64_t align_bits = 0;
  bool has_planes = false;  // some tile has nplanes > 1
  bool staged = false;      // eligible for the TMA-staged fan-out kernel when 16-byte aligned
  int max_fanout = 0;       // largest destination group
  int64_t tile_bytes = 0;   // source bytes of all tiles
  int64_t write_bytes = 0;  // bytes written: each tile's bytes times its replicas
  int64_t long_row_bytes = 0;  // ... of those in rows of at least 512 bytes (runs included)
  int64_t wide_row_bytes = 0;  // ... of those in rows of at least 8 KiB (runs included)
  int64_t narrow_row_bytes = 0;  // ... of those in rows under kNarrowRow bytes
  int64_t total_units() const { return prefix.empty() ? 0 : prefix.back(); }
  // transpose blocks (narrow innermost pieces grouped by shared rows)
  std::vector<reshard_tblock_t> tblocks;
  std::vector<reshard_tseg_t> tsegs;
  // OR of every block's row length and wide offset and every segment's width,
  // column and narrow offset (with the buffers' addresses: the element width)
  uint64_t talign_bits = 0;
  bool tscatter = false;  // some transpose block scatters (wide source -> narrow destinations)
  const reshard_tblock_t* d_tblocks = nullptr;
  const reshard_tseg_t* d_tsegs = nullptr;
};

// ------------------------------------------------------------ planner pieces
// (planner.cpp), shared with the multi-GPU partition (partition.cpp).

// Box (global offset + local shape) of one flat rank of a layout: Shard(d) on a
// mesh dim of size k splits the current local extent n of dim d into
// torch.chunk pieces of ceil(n/k); mesh dims apply in order.
void resolve_rank(int32_t nd, const int64_t* gshape, const Layout& L, int64_t rank, Box* b);
int64_t box_volume(int32_t nd, const Box& b);
// Ranks holding one identical, non-empty box (replicas), ranks ascending.
struct Class {
  Box box;
  std::vector<int64_t> ranks;
  int64_t volume = 0;
};
// The classes of a layout, leaving out the ranks marked in `gone` (may be empty).
std::vector<Class> classes_of(int32_t nd, const Layout& L, const std::vector<uint8_t>& gone);
struct Dim {
  int64_t e, ss, ds;  // extent, source stride, destination stride (elements)
};
void row_major_strides(int32_t nd, const int64_t* shp, int64_t* st);
// Appends to P the tiles copying a box of extents e[nd] (elements) that starts
// at element src_base / dst_base of buffers with strides sst / dst (elements),
// from buffer src_buf to destination group `group` (fanout = its replicas).
void emit_box(Program& P, uint16_t src_buf, uint16_t group, int32_t nd, const int64_t* e,
              int64_t src_base, const int64_t* sst, int64_t dst_base, const int64_t* dstr,
              int64_t eb, int64_t fanout = 1);
// Sorts P's tiles by destination and fills its prefix and summary fields.
void finish_program(Program& P);
int64_t tile_bytes(const reshard_tile_t& t);

// Narrow pieces (bytes per row) below this may go through transpose blocks
// (the planner's rule narrows it further), and a block holds at most this many
// bytes of wide rows in shared memory.
constexpr int64_t kTransposeMaxWidth = 129;
constexpr int64_t kTransposeBlockBytes = 20 * 1024;
// Blocks a transpose group aims for (smaller blocks when the group is small).
constexpr int64_t kTransposeMinBlocks = 128;
// Most segments one transpose group may have (the kernel stages them in shared memory).
constexpr int64_t kTransposeMaxSegs = 128;
// Most narrow replica pointers one scatter block may address.
constexpr int64_t kTransposeMaxReplicaPtrs = 512;

}  // namespace rs

struct reshard_plan_s {
  uint64_t magic = 0;
  int32_t ndim = 0;
  int64_t gshape[RESHARD_MAX_TENSOR_NDIM] = {};
  int32_t elem_bytes = 0;
  rs::Layout src, dst;
  rs::Program prog[rs::kNumPrograms];
  reshard_stats_t stats = {};
  // in-place plans: source rank s lives inside destination rank alias_dst[s]
  // (-1: separate buffer) at byte offset alias_off[s]
  bool inplace = false;
  std::vector<int64_t> alias_dst, alias_off;
  // ranks left out (a membership change): src_gone[s] / dst_gone[d] = 1; empty
  // when none.  A gone source is never read, a gone destination never written.
  std::vector<uint8_t> src_gone, dst_gone;
  // device binding (set once by upload_plan, under upload_mu)
  std::mutex upload_mu;
  int device = -1;
  void* d_mem = nullptr;
  int num_sms = 0;
  int blocks_per_sm = 0;
};

namespace rs {

// Host side shared by the plan and batch entry points (planner.cpp).
reshard_status_t upload_plan(reshard_plan_s* plan);
reshard_status_t buffer_table(reshard_plan_s* plan, const void* const* src_ptrs,
                              void* const* dst_ptrs, void* scratch,
                              std::vector<unsigned char*>* bufs);
// The same checks, into a caller-owned array of `capacity` entries (no heap use).
reshard_status_t buffer_table(reshard_plan_s* plan, const void* const* src_ptrs,
                              void* const* dst_ptrs, void* scratch, unsigned char** out,
                              int64_t capacity);
bool plan_live(const reshard_plan_s* plan);

// Error reporting (thread-local message).
reshard_status_t fail(reshard_status_t st, const std::string& msg);

// Kernel side (kernels.cu).  Launches one program over the buffer table
// bufs[nbufs] on `stream`.  Returns OK when there is nothing to do.
reshard_status_t launch_program(const reshard_plan_s* plan, const Program& p,
                                unsigned char* const* bufs, int nbufs, void* stream);
// The read-once path of a plan: its FANOUT program, then (same stream) its
// REPLICATE program when some destination classes are assembled in one replica.
reshard_status_t launch_fanout(const reshard_plan_s* plan, unsigned char* const* bufs, int nbufs,
                               void* stream);
// Same, with the program's tables at explicit device addresses (no uploaded plan).
reshard_status_t launch_program_tables(const Program& p, const reshard_tile_t* d_tiles,
                                       const int64_t* d_prefix, const uint32_t* d_goff,
                                       const uint16_t* d_gbuf, int num_sms,
                                       unsigned char* const* bufs, int nbufs, void* stream);
// The copy path an execution of `prog` with buffer table bufs[nbufs] takes
// (host-side decision, no device access).  allow_tma_fanout: false for the
// allocation-free entry point, whose programs never use the TMA fan-out.
struct Dispatch {
  int path = RESHARD_PATH_NONE;  // reshard_path_t
  int w_log2 = 0;                // widest common access, log2 bytes
  int kidx = 0;                  // copy-kernel table index (kernels.cu)
  int narrow = 0;                // 1: the variant for mostly narrow rows
  uint32_t flags = 0;            // kFlag* bits for the kernel
};
Dispatch decide(const Program& prog, unsigned char* const* bufs, int nbufs, bool allow_tma_fanout);
// TMA-staged fan-out (bulk_fanout.cu) for a 16-byte-aligned program.
reshard_status_t launch_fanout_staged(const reshard_plan_s* plan, const KernelParams& kp,
                                      const Program& prog, void* stream);
// TMA-staged realigning copy (realign_staged.cu) for a program that is not
// 16-byte aligned, on a grid of num_sms x its resident CTAs per SM.
reshard_status_t launch_realign_staged(int num_sms, const KernelParams& kp, const Program& prog,
                                       void* stream);
// A work-queue slot {next piece, CTAs finished} of the current device for one
// launch on `stream`; the launch's last CTA puts it back to zero.  Launches on one
// stream run in turn and share the stream's slot; a slot passes to another stream
// once its last launch has finished (an event recorded at release tells), or, when
// no slot is idle, the new stream first waits for the least recently used slot's
// last launch.  A launch being captured into a CUDA graph gets a slot of its own
// for good (bulk_fanout.cu); UNSUPPORTED when a device's slots for captured
// launches run out.  Every acquire is followed by one release after the launch
// (launched = whether the launch was enqueued).
struct QueueSlot {
  unsigned int* addr = nullptr;
  int dev = -1;
  int idx = -1;  // stream slot index, -1 for a captured launch
};
reshard_status_t work_queue_acquire(void* stream, QueueSlot* slot);
reshard_status_t work_queue_release(const QueueSlot& slot, void* stream, bool launched);
// The pieces a work queue hands out, in order: pieces of `big` units up to unit
// `split` (a multiple of big), then pieces of `small` units up to `total`, so
// that the last pieces taken are short and the CTAs of a launch finish close
// together.
struct PieceSchedule {
  int64_t total, big, split, small;
  RS_HOST_DEVICE int64_t count() const { return split / big + (total - split + small - 1) / small; }
  // Units [*u0, *u1) of piece i < count().
  RS_HOST_DEVICE void range(int64_t i, int64_t* u0, int64_t* u1) const {
    const int64_t nbig = split / big;
    if (i < nbig) {
      *u0 = i * big;
      *u1 = *u0 + big;
    } else {
      *u0 = split + (i - nbig) * small;
      *u1 = *u0 + small < total ? *u0 + small : total;
    }
  }
};
// The queue pieces for a program of total_units units that reads tile_bytes
// and writes write_bytes, on a grid of `grid` CTAs: big pieces of about 32 KiB
// read, at least 8 per CTA, but no less than min_piece_bytes while every CTA
// still gets one; the last two rounds of the grid in pieces a quarter that
// size, but of at least 40 KiB read plus written and still no less than
// min_piece_bytes (bulk_fanout.cu).
PieceSchedule work_queue_schedule(int64_t total_units, int64_t tile_bytes, int64_t write_bytes,
                                  int64_t grid, int64_t min_piece_bytes);
// Device address of the status word that bounded waits report into (bulk_fanout.cu).
reshard_status_t device_status_word(unsigned int** status);
// Transpose blocks of a program (transpose.cu); no-op when it has none.
reshard_status_t launch_transposes(const reshard_plan_s* plan, const Program& prog,
                                   unsigned char* const* bufs, int nbufs, uint32_t flags,
                                   void* stream);
// Occupancy of the copy kernel on the current device (blocks per SM).
reshard_status_t copy_kernel_occupancy(int* blocks_per_sm);

}  // namespace rs
