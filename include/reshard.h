/*
 * reshard.h -- C ABI of libreshard.so, a single-GPU DTensor-to-DTensor reshard.
 *
 * A global tensor laid out as M source shards (a device mesh plus one
 * Shard(dim) / Replicate placement per mesh dim) is rewritten into N
 * destination shards of another layout.  Only the intersections of source and
 * destination shard boxes are moved; the full tensor is never materialised on
 * the reshard path.  All shard buffers live in the memory of the current CUDA
 * device: every source or destination "rank" is simply its own device buffer.
 *
 * Defining passages ("Accelerating Reinforcement Learning Weight Refit with the
 * Reshard Collective", as summarised by the pages cited below):
 *  - news.bpdata.com, section "A megkozelites: refit mint DTensor-to-DTensor
 *    reshard": a DTensor is a global shape, a device mesh and placements
 *    (sharded or replicated); a destination shard can be built from parts of
 *    several source shards, and a replicated weight is available at several
 *    sources.
 *  - news.bpdata.com, section "A Reshard kollektiv kommunikacio": one call is
 *    given the source and destination DTensor descriptions; the library first
 *    determines the exact intersections of source and destination shards, then
 *    maps the transfers, sending each contribution once and letting replicas
 *    assemble their shard locally.
 *  - techfeed.io, section "Reshard Collective: DTensor-to-DTensor": the call is
 *    made once from the application, like all-reduce or all-gather, and the
 *    library derives the transfer pattern.
 *
 * Conventions shared by every entry point
 *  - Ranks are flat, row-major coordinates on their mesh.  Source and
 *    destination ranks are distinct buffers even when the meshes are equal.
 *  - A local shard is a contiguous row-major array of its local shape.
 *  - Uneven splits follow torch.chunk: Shard(d) on a mesh dim of size k splits
 *    the current local extent n of tensor dim d into chunks of ceil(n/k);
 *    trailing ranks get short or EMPTY shards.  Several mesh dims sharding the
 *    same tensor dim nest in mesh-dim order (mesh dim 0 outermost).
 *  - The reshard is a bit copy: the element size comes from the dtype, no
 *    value is converted, NaN payloads and -0 survive.
 *  - Every call returns a reshard_status_t; none aborts, traps or prints.  On
 *    failure reshard_last_error() describes the cause.
 *  - The caller owns every device buffer and stream.  Execution entry points
 *    enqueue work on `stream` (a cudaStream_t, NULL = legacy default stream)
 *    and return without synchronising; buffers must stay alive until that
 *    work has completed.  Pointer arrays are read during the call only.
 *  - Source replicas must hold identical bytes (they are replicas); which
 *    replica supplies a region is the planner's choice.
 */
#ifndef RESHARD_H_
#define RESHARD_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define RESHARD_MAX_TENSOR_NDIM 4
#define RESHARD_MAX_MESH_NDIM 4
/* Largest M + N (+1 for the scratch buffer) one execution call accepts. */
#define RESHARD_MAX_EXEC_BUFFERS 1024
/* Largest M or N plan creation accepts (planner-only use may exceed the above). */
#define RESHARD_MAX_RANKS 65000

typedef enum reshard_status {
  RESHARD_OK = 0,
  RESHARD_ERR_INVALID_ARG = 1, /* null pointer, bad enum, negative size, ... */
  RESHARD_ERR_UNSUPPORTED = 2, /* valid request outside what this library does */
  RESHARD_ERR_SHAPE = 3,       /* layout inconsistent with the tensor shape */
  RESHARD_ERR_CUDA = 4,        /* a CUDA runtime call failed */
  RESHARD_ERR_NO_MEMORY = 5,   /* host or device allocation failed */
  RESHARD_ERR_BAD_HANDLE = 6   /* plan is NULL, destroyed or never created */
} reshard_status_t;

/* Element types.  Only the element size matters (bit copy). */
typedef enum reshard_dtype {
  RESHARD_U8 = 0,   /* 1 byte  */
  RESHARD_BF16 = 1, /* 2 bytes */
  RESHARD_FP16 = 2, /* 2 bytes */
  RESHARD_FP32 = 3, /* 4 bytes */
  RESHARD_I32 = 4,  /* 4 bytes */
  RESHARD_FP64 = 5, /* 8 bytes */
  RESHARD_I64 = 6   /* 8 bytes */
} reshard_dtype_t;

/* Placement of a tensor on one mesh dim (DTensor's Replicate / Shard(dim)).
 * Partial (pending-reduction) placements are not part of the method. */
typedef enum reshard_placement_kind {
  RESHARD_REPLICATE = 0,
  RESHARD_SHARD = 1
} reshard_placement_kind_t;

typedef struct reshard_placement {
  int32_t kind; /* reshard_placement_kind_t */
  int32_t dim;  /* tensor dim for RESHARD_SHARD, ignored for RESHARD_REPLICATE */
} reshard_placement_t;

typedef struct reshard_mesh {
  int32_t ndim;                           /* 1..RESHARD_MAX_MESH_NDIM */
  int64_t shape[RESHARD_MAX_MESH_NDIM];   /* sizes >= 1; ranks = product */
} reshard_mesh_t;

typedef struct reshard_plan_s* reshard_plan_t;
typedef struct reshard_batch_s* reshard_batch_t;
typedef struct reshard_refit_s* reshard_refit_t;

/* Which copy kernel an execution uses. */
typedef enum reshard_kernel {
  /* Read-once fan-out (default): each region is read once from one source
   * replica and written to every destination replica that needs it.  HBM
   * traffic = global bytes G (read) + destination bytes D (write).  Where the
   * planner assembles a destination shard in one replica first (program
   * RESHARD_PROGRAM_REPLICATE: many replicas fed by pieces off the 16-byte
   * grid), a second launch on the same stream copies it to the other replicas,
   * and that shard is read once more. */
  RESHARD_KERNEL_FANOUT = 0,
  /* Plain box copy: one copy per (region, destination replica); the source
   * is re-read for every replica.  HBM traffic = D (read) + D (write). */
  RESHARD_KERNEL_BOXCOPY = 1
} reshard_kernel_t;

/* Copy path of an execution's tiles (reshard_plan_path); transpose blocks,
 * when a program has any, always run in their own kernel after the tiles. */
typedef enum reshard_path {
  RESHARD_PATH_NONE = 0,        /* the program has no tiles */
  RESHARD_PATH_VECTOR = 1,      /* element-width vector kernel (1..16-byte accesses) */
  RESHARD_PATH_TMA_FANOUT = 2,  /* 16-byte aligned: TMA bulk copies through shared memory */
  RESHARD_PATH_REALIGN = 3,     /* aligned 16-byte loads and stores, bytes realigned in registers */
  RESHARD_PATH_STAGED = 4,      /* TMA-staged realigning copy, stores from registers */
  RESHARD_PATH_STAGED_BULK = 5  /* TMA-staged realigning copy, bulk stores to every replica */
} reshard_path_t;

/* Copy programs a plan holds (for inspection and for the CPU test executor). */
typedef enum reshard_program {
  RESHARD_PROGRAM_FANOUT = 0,  /* reshard, read-once fan-out */
  RESHARD_PROGRAM_BOXCOPY = 1, /* reshard, one copy per destination replica */
  RESHARD_PROGRAM_GATHER = 2,  /* gather-and-broadcast step 1: shards -> full */
  RESHARD_PROGRAM_SLICE = 3,   /* gather-and-broadcast step 2: full -> shards */
  RESHARD_PROGRAM_REPLICATE = 4 /* reshard, second step of FANOUT: a destination shard that the
                                   first step assembled in one replica, copied as one run to
                                   the class's other replicas (empty for most plans) */
} reshard_program_t;

/* Planner and traffic statistics of one plan (all byte counts exact). */
typedef struct reshard_stats {
  int64_t global_bytes;        /* G: bytes of the global tensor */
  int64_t src_bytes;           /* sum of all source shard bytes (replicas included) */
  int64_t dst_bytes;           /* D: sum of all destination shard bytes (replicas included) */
  int64_t n_src_ranks, n_dst_ranks;
  int64_t n_src_classes;       /* distinct non-empty source boxes */
  int64_t n_dst_classes;       /* distinct non-empty destination boxes (fan-out groups) */
  int64_t n_regions;           /* source-class x destination-class intersections moved */
  int64_t region_bytes;        /* sum of region bytes (= G for a complete layout) */
  int64_t n_tiles[4];          /* tiles per reshard_program_t */
  int64_t fanout_read_bytes, fanout_write_bytes;    /* HBM bytes of RESHARD_KERNEL_FANOUT */
  int64_t boxcopy_read_bytes, boxcopy_write_bytes;  /* HBM bytes of RESHARD_KERNEL_BOXCOPY */
  int64_t gb_read_bytes, gb_write_bytes;            /* HBM bytes of gather_broadcast_execute */
  int64_t max_replica_read_bytes;  /* busiest source replica's bytes read (fan-out plan) */
  int64_t max_fanout;          /* largest number of destination replicas of one box */
  int64_t planner_ns;          /* wall time of reshard_plan_create */
  int64_t inplace_bytes;       /* destination bytes already in place (in-place plans), not written */
  int64_t assembled_classes;   /* destination classes assembled in one replica, then replicated */
  int64_t n_replicate_tiles;   /* tiles of RESHARD_PROGRAM_REPLICATE */
} reshard_stats_t;

/*
 * One copy descriptor ("tile") as the kernels execute it, exposed read-only
 * for inspection and tests.  A tile copies nplanes x nrows rows of row_bytes
 * from its source buffer to the same local place in every buffer of its
 * destination group.  Byte offsets and strides are relative to the start of
 * the buffers.  Buffer indices: [0, M) source ranks, [M, M+N) destination
 * ranks, M+N the gather-and-broadcast scratch.
 */
typedef struct reshard_tile {
  int64_t src_off, dst_off;                   /* bytes, first row of plane 0 */
  int64_t src_row_stride, dst_row_stride;     /* bytes between rows */
  int64_t src_plane_stride, dst_plane_stride; /* bytes between planes */
  uint32_t row_bytes;                         /* contiguous bytes per row */
  uint32_t nrows;                             /* rows per plane */
  uint32_t nplanes;
  uint16_t src_buf;                           /* buffer index of the source */
  uint16_t dst_group;                         /* destination group index */
} reshard_tile_t;

/*
 * Transpose blocks (read-only view, for inspection and tests).  When a tensor is
 * sharded on its innermost dim into narrow pieces (under 64 bytes per row) on
 * one side and into whole rows on the other, per-piece copies would write a few
 * bytes per row.  The planner then groups the pieces that share their rows: a
 * block is nrows consecutive rows of row_bytes on the "wide" side (one buffer
 * or destination group, contiguous) and seg_count narrow segments, each a
 * dense run of nrows x width bytes on its own buffer or destination group,
 * occupying bytes [col, col + width) of every wide row.  The kernel assembles
 * or splits the rows in shared memory, so both sides move contiguous bytes.
 *   direction 0 (gather):  narrow sources -> wide destination group;
 *   direction 1 (scatter): wide source -> narrow destination groups.
 * flags: RESHARD_TBLOCK_SAME_SHAPE when the block has the shape of the block
 * before it in the program (same wide side, direction, row length, rows, and
 * segments of the same widths, columns and narrow sides in the same order; only
 * the offsets differ), so a kernel may keep what it derived from that shape;
 * RESHARD_TBLOCK_FOLLOWS (with SAME_SHAPE) when moreover its wide rows and every
 * narrow range start right where the previous block's end (offsets advanced by
 * nrows x row_bytes and nrows x width).
 */
#define RESHARD_TBLOCK_SAME_SHAPE 1u
#define RESHARD_TBLOCK_FOLLOWS 2u
typedef struct reshard_tblock {
  int64_t wide_off;    /* bytes: row 0 of the block in the wide buffer(s) */
  uint32_t row_bytes;  /* wide row length */
  uint32_t nrows;
  uint32_t seg_begin, seg_count;
  uint16_t wide;       /* gather: destination group; scatter: source buffer index */
  uint16_t direction;  /* 0 gather, 1 scatter */
  uint32_t flags;      /* RESHARD_TBLOCK_* bits */
} reshard_tblock_t;

typedef struct reshard_tseg {
  int64_t narrow_off;  /* bytes: row 0 of the block in the narrow buffer(s) */
  uint32_t width;      /* bytes per row */
  uint32_t col;        /* byte offset of the segment inside a wide row */
  uint16_t narrow;     /* gather: source buffer index; scatter: destination group */
  uint16_t pad16;
  uint32_t pad32;
} reshard_tseg_t;

/*
 * Plan a reshard of one tensor (steps: resolve both layouts, intersect every
 * source box with every destination box, pick one source replica per region
 * balancing bytes read across replicas, collapse contiguous dims into copy
 * descriptors, group destination replicas for fan-out, sort by destination).
 * Host only: needs no GPU and touches no device memory.
 *
 * global_shape  [tensor_ndim] extents >= 0 (1 <= tensor_ndim <= 4)
 * dtype         element type (sets the element size)
 * src_mesh, src_placements[src_mesh->ndim]: source layout
 * dst_mesh, dst_placements[dst_mesh->ndim]: destination layout
 * out_plan      receives the plan; release it with reshard_plan_destroy().
 * Errors: INVALID_ARG (null/ranges/enums), UNSUPPORTED (ndim or ranks beyond
 * the limits above), NO_MEMORY.
 */
reshard_status_t reshard_plan_create(const int64_t* global_shape, int32_t tensor_ndim,
                                     reshard_dtype_t dtype, const reshard_mesh_t* src_mesh,
                                     const reshard_placement_t* src_placements,
                                     const reshard_mesh_t* dst_mesh,
                                     const reshard_placement_t* dst_placements,
                                     reshard_plan_t* out_plan);

/*
 * In-place plan (HybridFlow's 3D-HybridEngine: siliconandsystems.com HybridFlow
 * summary, section on moving the actor without redundant copies -- generation
 * ranks are assigned at a stride so that each rank's generation shard contains
 * its own training shard, and no weight is held twice).  src_alias[s] names the
 * destination rank whose buffer ALREADY HOLDS source shard s (or -1 when s has
 * a buffer of its own).  Source rank s's box must lie inside that destination
 * box and form one contiguous range of its row-major local layout (leading
 * dims of extent 1, one partial dim, trailing dims full); otherwise
 * RESHARD_ERR_SHAPE.  The plan then skips every copy whose bytes are already in
 * place: a region is written only to the destination replicas that do not
 * hold it (reshard_stats_t.inplace_bytes counts the bytes skipped).
 * Executions of such a plan require src_ptrs[s] == dst_ptrs[src_alias[s]] +
 * the offset reported by reshard_plan_alias() for every aliased s
 * (RESHARD_ERR_INVALID_ARG otherwise); source and destination buffers may then
 * overlap exactly in that way, and no copy writes a byte that another copy
 * of the same execution reads.  Other arguments and errors as
 * reshard_plan_create.
 */
reshard_status_t reshard_plan_create_inplace(const int64_t* global_shape, int32_t tensor_ndim,
                                             reshard_dtype_t dtype, const reshard_mesh_t* src_mesh,
                                             const reshard_placement_t* src_placements,
                                             const reshard_mesh_t* dst_mesh,
                                             const reshard_placement_t* dst_placements,
                                             const int64_t* src_alias, reshard_plan_t* out_plan);

/* Destination rank (-1 if none) and byte offset at which source rank src_rank lives in an
 * in-place plan.  Errors: BAD_HANDLE, INVALID_ARG. */
reshard_status_t reshard_plan_alias(reshard_plan_t plan, int64_t src_rank, int64_t* dst_rank,
                                    int64_t* byte_offset);

/*
 * Copy the plan's descriptor tables to the CURRENT device (one cudaMalloc and
 * one synchronous cudaMemcpy) and bind the plan to it.  Executions call this
 * themselves on first use; call it explicitly to keep allocation out of the
 * first execution, and always before capturing an execution in a CUDA graph.
 * Errors: BAD_HANDLE, CUDA (no device, copy failed), NO_MEMORY,
 * INVALID_ARG (plan already bound to a different device).
 */
reshard_status_t reshard_plan_upload(reshard_plan_t plan);

/*
 * The reshard itself (news.bpdata.com, section "A Reshard kollektiv
 * kommunikacio"): every destination shard receives exactly the intersections
 * of its box with the source boxes, each region read once and fanned out to
 * all destination replicas.  Equivalent to
 * reshard_execute_ex(plan, src_ptrs, dst_ptrs, RESHARD_KERNEL_FANOUT, stream).
 *
 * src_ptrs[M]  device pointers of the source shards (NULL allowed only for an
 *              empty shard).  dst_ptrs[N] likewise for the destinations.
 * Destination buffers must not overlap each other or any source buffer
 * (except as declared for in-place plans).  Once the plan is uploaded and one
 * execution has run on the device, executions can be recorded into a CUDA graph
 * by stream capture and replayed; the graph keeps the buffer addresses.
 * Errors: BAD_HANDLE, INVALID_ARG (null pointer for a non-empty shard),
 * UNSUPPORTED (M + N + 1 > RESHARD_MAX_EXEC_BUFFERS, or the device's 3072
 * work-queue slots for launches captured into CUDA graphs are used up: each
 * captured launch keeps one for good), CUDA (launch failed).  Eager executions
 * on any number of streams are supported: the 1024 per-stream slots pass from a
 * stream to another once the slot's last launch has finished (when none has, the
 * new stream first waits for the least recently used slot's last launch).
 */
reshard_status_t reshard_execute(reshard_plan_t plan, const void* const* src_ptrs,
                                 void* const* dst_ptrs, void* stream);

/* reshard_execute with an explicit choice of copy kernel (reshard_kernel_t). */
reshard_status_t reshard_execute_ex(reshard_plan_t plan, const void* const* src_ptrs,
                                    void* const* dst_ptrs, int32_t kernel, void* stream);

/*
 * The conventional refit path, kept as the baseline (news.bpdata.com, section
 * "Miert problema a sulyrefit az RL post-training soran?"; techfeed.io, section
 * on the payload being twice the model size): all-gather the full parameter,
 * broadcast it, and let every destination keep its slice.  On one GPU the
 * broadcast is free, so this is: (1) every source region is written into
 * `full_scratch` (the global tensor, row-major), then (2) every destination
 * rank copies its own box out of it.  Same destination bytes as
 * reshard_execute.  HBM traffic = 2G + 2D.
 *
 * full_scratch  device buffer of at least G bytes, owned by the caller; its
 *               contents on return are the global tensor.
 * scratch_bytes its size in bytes.
 * Errors: as reshard_execute, plus INVALID_ARG when scratch_bytes < G or
 * full_scratch is NULL for a non-empty tensor.
 */
reshard_status_t gather_broadcast_execute(reshard_plan_t plan, const void* const* src_ptrs,
                                          void* const* dst_ptrs, void* full_scratch,
                                          size_t scratch_bytes, void* stream);

/*
 * Status word of the current device's copy kernels (no counterpart on the pages:
 * failure detection of this library).  The TMA-staged fan-out kernel bounds
 * every wait on its shared-memory barriers; a wait that runs out (which a
 * correct run never does) records a nonzero code here instead of hanging or
 * trapping, and the kernel returns.  Codes: 0 none, 1 producer wait, 2 consumer
 * wait, 3 self-test.  Synchronous (reads device memory with cudaMemcpy);
 * `clear` != 0 resets the word to 0 after reading.  Errors: INVALID_ARG, CUDA.
 */
reshard_status_t reshard_device_status(int32_t clear, uint32_t* status);

/*
 * Launch, on `stream`, one CTA that waits on a shared-memory barrier nobody
 * will ever arrive at, with the same bounded wait as the copy kernels but a
 * limit of `polls` polls (1..2^20).  After the stream completes,
 * reshard_device_status() reports code 3 and the device remains usable.  For
 * tests of the failure path.  Errors: INVALID_ARG, CUDA.
 */
reshard_status_t reshard_selftest_wait_timeout(uint32_t polls, void* stream);

/* Sizes of the static device arrays used by gather_broadcast_execute_static. */
#define RESHARD_STATIC_SCRATCH_BYTES (64ull << 20) /* largest global tensor: 64 MiB */
#define RESHARD_STATIC_TABLE_BYTES (1ull << 20)    /* gather + slice descriptor tables */

/*
 * gather_broadcast_execute without any allocation.  The write-ups have no
 * counterpart of this entry point; it exists for callers that cannot call
 * cudaMalloc: an inference engine whose memory pool has already claimed the
 * device memory it may use, a caller in a latency-critical path that must not
 * incur the implicit device synchronisation cudaMalloc/cudaFree can cause, or
 * code that owns no allocator at all (a plugin handed only its input and output
 * buffers).  Such callers cannot provide the full-tensor scratch nor the
 * plan's device tables that the other entry points allocate.
 *
 * Instead, the scratch (RESHARD_STATIC_SCRATCH_BYTES) and the descriptor tables
 * (RESHARD_STATIC_TABLE_BYTES) live in file-scope static device arrays of the
 * library: every GPU on which the library's device code is loaded holds those
 * 65 MiB until the process exits.  The caller passes only the source and
 * destination pointers (as for gather_broadcast_execute) and the stream; the
 * result is the same.  The plan need not be uploaded.
 *
 * The first call on a device looks up the arrays' device addresses
 * (cudaGetSymbolAddress) with that device current.  Each call copies the plan's
 * tables from host memory into the static array with cudaMemcpyAsync on
 * `stream` and then launches the gather and slice kernels on `stream`.  No part of the arrays needs to start at
 * zero: the gather writes every byte of the global tensor before the slice reads
 * it, and the tables are rewritten by every call.
 *
 * All calls share the arrays and each call overwrites the previous contents:
 * calls that can overlap on the GPU (different streams without ordering between
 * them, or several host threads) race and produce wrong results.  Calls on one
 * stream are safe because the stream orders each call's table copy after the
 * previous call's kernels.  No cudaMalloc, cudaFree or other allocating library
 * routine is called.  The pointers are checked as for every other execution: a
 * NULL pointer is accepted for an empty shard and for a rank that an excluded
 * plan (reshard_plan_exclude) leaves out, and in-place plans must pass aliased
 * source pointers.
 *
 * Errors: as gather_broadcast_execute, plus UNSUPPORTED when the global tensor
 * exceeds RESHARD_STATIC_SCRATCH_BYTES or the gather + slice tables exceed
 * RESHARD_STATIC_TABLE_BYTES (use gather_broadcast_execute with a caller-owned
 * scratch then), CUDA when the symbol lookup or the table copy fails.
 */
reshard_status_t gather_broadcast_execute_static(reshard_plan_t plan, const void* const* src_ptrs,
                                                 void* const* dst_ptrs, void* stream);

/*
 * Whole-model batching: the fan-out reshards of several plans (e.g. every
 * feed-forward weight of a model) with the plans that take the TMA fan-out as
 * ONE kernel launch: their copy descriptors are concatenated over a combined
 * buffer table, and the kernel's work queue spreads the work evenly over the
 * GPU with no launch boundary between tensors.  Every other plan runs on its
 * own, as reshard_execute runs it (see reshard_batch_classes).  The
 * pages route the feed-forward projections (most of the parameters) through
 * the Reshard collective and the small irregular weights through
 * gather-and-broadcast (news.bpdata.com, section "Integracio es hibrid megoldas
 * a NeMo RL-ben"); a batch is the unit for the first group.
 *
 * reshard_batch_create: plans[nplans] stay owned by the caller and must outlive
 * the batch (executions check them).  TMA fan-out plans that together have
 * more ranks (M + N each) than one launch can address (RESHARD_MAX_EXEC_BUFFERS)
 * go to several launches; a plan that alone has more (which no reshard_execute
 * could run either) makes the call fail with UNSUPPORTED.
 * Errors: INVALID_ARG, BAD_HANDLE, UNSUPPORTED, NO_MEMORY.
 */
reshard_status_t reshard_batch_create(const reshard_plan_t* plans, int32_t nplans,
                                      reshard_batch_t* out_batch);

/*
 * Execute every plan of the batch: src_ptrs[i] and dst_ptrs[i] are plan i's
 * pointer arrays, exactly as for reshard_execute (in-place plans included).
 * The merged TMA fan-out plans are one launch (its descriptor tables are
 * uploaded on first use, like a plan's) when all their buffers are 16-byte
 * aligned (torch allocations are); otherwise they too run one by one, each
 * with its own kernel.  All pointer arrays are checked before anything is
 * launched.  Errors: as reshard_execute.
 */
reshard_status_t reshard_batch_execute(reshard_batch_t batch, const void* const* const* src_ptrs,
                                       void* const* const* dst_ptrs, void* stream);

/*
 * The launch classes of a batch, in the order they run on the stream: one
 * for the merged TMA fan-out plans (more if their ranks overflow a launch's
 * buffer table), one for each other plan.  *nclasses (may be NULL) receives
 * their number, plan_class[nplans] (may be NULL) the class of each plan, -1
 * for a plan with nothing to copy.  Errors: BAD_HANDLE.
 */
reshard_status_t reshard_batch_classes(reshard_batch_t batch, int32_t* nclasses, int32_t* plan_class);

/* Release a batch (not its plans).  Errors: BAD_HANDLE. */
reshard_status_t reshard_batch_destroy(reshard_batch_t batch);

/*
 * Whole-model refit with the pages' hybrid routing (news.bpdata.com, section
 * "Integracio es hibrid megoldas a NeMo RL-ben": the feed-forward projections,
 * about 95% of the parameters, go through the Reshard path; smaller special
 * weights such as QKV projections through gather-and-broadcast).  A refit
 * holds plans[nplans] (owned by the caller, checked at every execution) and a
 * route for each; one reshard_refit_execute then runs the whole model on one
 * stream: the reshard group first (one batch launch with RESHARD_REFIT_BATCH,
 * else one launch per plan), then every gather-and-broadcast plan in turn
 * through one shared scratch buffer (stream order makes the reuse safe).
 *
 * Routes: RESHARD_ROUTE_RESHARD, RESHARD_ROUTE_GATHER_BROADCAST, or
 * RESHARD_ROUTE_AUTO, which on one GPU always resolves to the reshard (it moves
 * G + D bytes in one launch against 2G + 2D in two); routes == NULL means AUTO
 * for every plan.  The split therefore only changes where it is asked for.
 */
typedef enum reshard_route {
  RESHARD_ROUTE_AUTO = 0,
  RESHARD_ROUTE_RESHARD = 1,
  RESHARD_ROUTE_GATHER_BROADCAST = 2
} reshard_route_t;

/* reshard_refit_create flag: batch the reshard group into one launch. */
#define RESHARD_REFIT_BATCH 1u
/* reshard_refit_create flag: spread the reshard group over
 * RESHARD_REFIT_NUM_LANES side streams of the current device, so that the
 * launches of independent tensors overlap (a launch of a small tensor fills few
 * SMs for a few microseconds, and each launch drains its last CTAs alone).  The
 * group is cut into units: one plan each, or, with RESHARD_REFIT_BATCH as well,
 * the plans that a batch concatenates into one launch form one unit (a batch of
 * their own) and every other plan is a unit of one.  Units go to the lanes
 * largest first, each to the lane with the fewest bytes so far.  reshard_refit_execute makes the lanes wait for the caller's stream,
 * launches every plan on its lane and makes the caller's stream wait for every
 * lane before the gather-and-broadcast group, so the call is ordered on the
 * caller's stream like the one-stream form and can be captured into a CUDA graph
 * from it.  The side streams are created at the first such refit of a device,
 * shared by all refits of that device and kept until the process exits;
 * executions of such refits are issued one at a time (one process-wide lock, so
 * that a lane taking part in one caller's CUDA-graph capture gets no other
 * execution's launches), and the refit must be executed with the device current
 * that it was created on (INVALID_ARG otherwise).  While one caller's stream
 * capture that took in a lanes execution is open, the side streams belong to it:
 * an execution from any other stream returns UNSUPPORTED until that capture
 * ends. */
#define RESHARD_REFIT_LANES 2u
#define RESHARD_REFIT_NUM_LANES 4

/* Errors: INVALID_ARG (no plans, unknown route or flag),
 * BAD_HANDLE (a plan is not live), UNSUPPORTED (RESHARD_REFIT_BATCH and the
 * reshard group exceeds one batch's buffer table), CUDA (LANES: creating the
 * side streams or events failed), NO_MEMORY. */
reshard_status_t reshard_refit_create(const reshard_plan_t* plans, const int32_t* routes,
                                      int32_t nplans, uint32_t flags, reshard_refit_t* out_refit);

/* Resolved routes (routes[nplans], may be NULL) and the scratch bytes that
 * reshard_refit_execute needs (the largest global tensor on the
 * gather-and-broadcast route; 0 when there is none).  Errors: BAD_HANDLE. */
reshard_status_t reshard_refit_info(reshard_refit_t refit, int32_t* routes, uint64_t* scratch_bytes);

/* src_ptrs[i] / dst_ptrs[i]: plan i's pointer arrays, as for reshard_execute.
 * scratch: device buffer of scratch_bytes >= the reshard_refit_info figure (may
 * be NULL when that is 0).  Errors: as reshard_execute and
 * gather_broadcast_execute; BAD_HANDLE when the refit or one of its plans is
 * gone.  On an error the calls already enqueued stay enqueued. */
reshard_status_t reshard_refit_execute(reshard_refit_t refit, const void* const* const* src_ptrs,
                                       void* const* const* dst_ptrs, void* scratch,
                                       size_t scratch_bytes, void* stream);

/* Release the refit (its batch too; the plans stay).  Errors: BAD_HANDLE. */
reshard_status_t reshard_refit_destroy(reshard_refit_t refit);

/*
 * Multi-GPU partition of one reshard (news.bpdata.com, section "A Reshard
 * kollektiv kommunikacio": each contribution crosses the network once, the
 * replicas are assembled inside the NVLink domain with a balanced exchange, and
 * the two stages are pipelined; techfeed.io, section on NVIDIA's NVLink
 * implementation: incoming data spread as evenly as possible over the replicas).
 *
 * reshard_partition_create cuts a plan by destination ownership.  src_gpu[M]
 * and dst_gpu[N] give the GPU (0..ngpus-1) of every source and destination
 * rank (ignored for ranks an excluded plan leaves out), gpu_domain[ngpus] the
 * NVLink domain of every GPU (any non-negative ids; GPUs with equal ids share a
 * domain).  Every GPU g then owns:
 *   - the LOCAL step: regions whose source replica is on g, copied to all of
 *     g's destination replicas of the region's class (one read, R writes);
 *   - per pipeline chunk c (0..nchunks-1), three steps around two rounds of
 *     messages:
 *       PACK c     stage-0 pieces g sends, copied from its source shards into
 *                  its send buffer;
 *       (stage 0)  the messages of stage 0 of chunk c;
 *       FORWARD c  stage-1 pieces g sends, copied from where they landed in
 *                  its receive buffer in stage 0 into its send buffer;
 *       (stage 1)  the messages of stage 1 of chunk c;
 *       UNPACK c   every piece g received in chunk c, copied from its receive
 *                  buffer to all of g's destination replicas of its class.
 * Routing: a region that g needs and holds in a local source shard is copied
 * locally; a domain that holds a source replica of a region gets it from one
 * inside the domain (stage 0), the least-loaded such GPU per piece; a domain
 * that holds none receives each piece ONCE across domains (stage 0; sender: the
 * least-loaded GPU holding a source replica, receiver: the least-loaded GPU of
 * the domain that needs it), and the receiver forwards it to the domain's other
 * GPUs that need it (stage 1).  Loads are bytes sent (senders) and received
 * (receivers), pieces taken largest first.  Regions that cross GPUs are cut
 * along their outermost dim into nchunks (1..64) pieces, piece i in pipeline
 * chunk i (regions with fewer rows than chunks: one piece per row, chunks taken
 * in turn), so every link's bytes split evenly over the chunks; with
 * nchunks > 1, chunk c uses slot c % 2 of the send and receive buffers.
 *
 * Messages are packed: all pieces from one GPU to another in one chunk and
 * stage form one contiguous, 16-byte-aligned range of the sender's send buffer
 * and of the receiver's receive buffer, pieces in the same order on both sides,
 * each piece row-major in its own box and 16-byte aligned.  The library moves
 * nothing between GPUs: the caller performs every message (NCCL send/recv, peer
 * copies; never multicast) between the steps.  A valid order on one stream:
 * LOCAL; PACK 0; stage 0 of chunk 0; FORWARD 0; then for c = 1..nchunks-1:
 * PACK c, stage 1 of chunk c-1 together with stage 0 of chunk c, UNPACK c-1,
 * FORWARD c; finally stage 1 of the last chunk and its UNPACK.  With a single
 * chunk: LOCAL, PACK 0, stage 0, FORWARD 0, stage 1, UNPACK 0.
 *
 * The partition is a host object (no device memory until a step runs) and is
 * the same on every process that builds it from the same plan and maps.
 * Errors: BAD_HANDLE, INVALID_ARG (null map, a GPU id out of range, a negative
 * domain, ngpus or nchunks out of range), UNSUPPORTED (in-place plans; M + N + 2
 * > RESHARD_MAX_EXEC_BUFFERS), NO_MEMORY.
 */
typedef struct reshard_partition_s* reshard_partition_t;

typedef enum {
  RESHARD_STEP_LOCAL = 0,
  RESHARD_STEP_PACK = 1,
  RESHARD_STEP_FORWARD = 2,
  RESHARD_STEP_UNPACK = 3
} reshard_step_t;

/* One message of one GPU: in chunk `chunk`, stage `stage` (0 or 1), this GPU
 * sends (dir 0) bytes [offset, offset + bytes) of its send buffer to GPU `peer`,
 * or receives (dir 1) them into [offset, offset + bytes) of its receive buffer
 * from `peer`.  Both ends of a message list the same byte count. */
typedef struct {
  int32_t chunk;
  int32_t stage;
  int32_t peer;
  int32_t dir;
  int64_t offset;
  int64_t bytes;
} reshard_xfer_t;

/* One GPU's share: the sizes of the send and receive buffers it must provide,
 * bytes it copies from local source shards (each region once), and payload
 * bytes (without padding) it sends and receives across domains (inter) and
 * inside its domain (intra). */
typedef struct {
  int64_t send_bytes;
  int64_t recv_bytes;
  int64_t local_bytes;
  int64_t sent_inter_bytes;
  int64_t sent_intra_bytes;
  int64_t recv_inter_bytes;
  int64_t recv_intra_bytes;
  int64_t n_xfers;
} reshard_partition_gpu_t;

/* The whole partition: destination bytes filled from a source shard on the same
 * GPU (each replica counted), payload bytes sent across domains (every piece at
 * most once per receiving domain) and inside domains, the largest per-GPU sent
 * and received payloads, pieces, messages and planning time. */
typedef struct {
  int32_t ngpus;
  int32_t ndomains;
  int32_t nchunks;
  int32_t nslots;
  int64_t local_bytes;
  int64_t inter_domain_bytes;
  int64_t intra_domain_bytes;
  int64_t max_gpu_send_bytes;
  int64_t max_gpu_recv_bytes;
  int64_t n_pieces;
  int64_t n_messages;
  int64_t planner_ns;
} reshard_partition_stats_t;

reshard_status_t reshard_partition_create(reshard_plan_t plan, const int32_t* src_gpu,
                                          const int32_t* dst_gpu, int32_t ngpus,
                                          const int32_t* gpu_domain, int32_t nchunks,
                                          reshard_partition_t* out_partition);

/* Whole-partition figures.  Errors: BAD_HANDLE, INVALID_ARG. */
reshard_status_t reshard_partition_stats(reshard_partition_t part, reshard_partition_stats_t* out);

/* One GPU's share.  Errors: BAD_HANDLE, INVALID_ARG. */
reshard_status_t reshard_partition_gpu(reshard_partition_t part, int32_t gpu,
                                       reshard_partition_gpu_t* out);

/* Read-only view of one GPU's messages, valid until the partition is destroyed,
 * sorted by (chunk, stage, dir, peer).  Errors: BAD_HANDLE, INVALID_ARG. */
reshard_status_t reshard_partition_transfers(reshard_partition_t part, int32_t gpu,
                                             const reshard_xfer_t** xfers, int64_t* n);

/* Read-only view of the copy program of one step (reshard_step_t; chunk is
 * ignored for LOCAL) of one GPU, as reshard_plan_program gives it.  Buffer
 * indices: source rank r = r, destination rank r = M + r, the receive buffer
 * M + N, the send buffer M + N + 1.  Errors: BAD_HANDLE, INVALID_ARG. */
reshard_status_t reshard_partition_program(reshard_partition_t part, int32_t gpu, int32_t step,
                                           int32_t chunk, const reshard_tile_t** tiles,
                                           int64_t* ntiles, const int64_t** unit_prefix,
                                           const uint32_t** group_offsets,
                                           const uint16_t** group_buffers, int64_t* ngroups);

/*
 * Launch one step of one GPU on `stream` (the current device).  src_ptrs[M] and
 * dst_ptrs[N] are indexed by rank; only the ranks on this GPU are read (a NULL
 * is accepted for ranks the step's GPU does not read or write; entries of ranks
 * on other GPUs are ignored).  recv_buf / send_buf: this GPU's buffers of at
 * least reshard_partition_gpu's recv_bytes / send_bytes (may be NULL when that
 * is 0).  The first launch of a step uploads its tables (one cudaMalloc and one
 * synchronous copy), binding that step to the current device.  Errors:
 * BAD_HANDLE, INVALID_ARG, CUDA.
 */
reshard_status_t reshard_partition_execute(reshard_partition_t part, int32_t gpu, int32_t step,
                                           int32_t chunk, const void* const* src_ptrs,
                                           void* const* dst_ptrs, void* recv_buf, void* send_buf,
                                           void* stream);

/* Release the partition and its device tables (the plan stays).  Errors: BAD_HANDLE. */
reshard_status_t reshard_partition_destroy(reshard_partition_t part);

/*
 * Local box of one rank (news.bpdata.com, section "A megkozelites": the DTensor
 * description fixes each rank's shard).  side 0 = source, 1 = destination.
 * shape[tensor_ndim], offset[tensor_ndim] receive the local shape and the
 * global offset; an empty dim reports offset = global extent (DTensor's
 * convention).  Errors: BAD_HANDLE, INVALID_ARG.
 */
reshard_status_t reshard_plan_local_shape(reshard_plan_t plan, int32_t side, int64_t rank,
                                          int64_t* shape, int64_t* offset);

/* Planner and traffic statistics.  Errors: BAD_HANDLE, INVALID_ARG. */
reshard_status_t reshard_plan_stats(reshard_plan_t plan, reshard_stats_t* out);

/*
 * Read-only view of one copy program (reshard_program_t) of the plan, valid
 * until the plan is destroyed: tiles[ntiles], unit_prefix[ntiles + 1] (the
 * kernels' work units; see reshard_tile_units), group_offsets[ngroups + 1]
 * and group_buffers[group_offsets[ngroups]] (destination buffer indices of
 * each group).  Any output pointer may be NULL.  Errors: BAD_HANDLE,
 * INVALID_ARG.
 */
reshard_status_t reshard_plan_program(reshard_plan_t plan, int32_t program,
                                      const reshard_tile_t** tiles, int64_t* ntiles,
                                      const int64_t** unit_prefix,
                                      const uint32_t** group_offsets,
                                      const uint16_t** group_buffers, int64_t* ngroups);

/*
 * Read-only view of a program's transpose blocks (see reshard_tblock_t), valid
 * until the plan is destroyed.  Only the FANOUT program has any.  Any output
 * pointer may be NULL.  Errors: BAD_HANDLE, INVALID_ARG.
 */
reshard_status_t reshard_plan_transposes(reshard_plan_t plan, int32_t program,
                                         const reshard_tblock_t** blocks, int64_t* nblocks,
                                         const reshard_tseg_t** segs, int64_t* nsegs);

/*
 * The copy path reshard_execute_ex(plan, src_ptrs, dst_ptrs, kernel, ...)
 * would take with these buffers, decided on the host exactly as an execution
 * decides it (from the tiles' offsets, strides and row lengths, the buffers'
 * addresses mod 16, the fan-out and the program's size); nothing is launched
 * and no device memory is touched, so any pointers that pass the execution's
 * argument checks may be given.  *path receives a reshard_path_t, *width the
 * widest access in bytes every tile allows (1..16).  Either output may be
 * NULL.  For the fan-out this is the path of the first launch; a REPLICATE
 * step, when the plan has one, is a plain run copy.  Errors: BAD_HANDLE,
 * INVALID_ARG (as reshard_execute_ex), UNSUPPORTED.
 */
reshard_status_t reshard_plan_path(reshard_plan_t plan, const void* const* src_ptrs,
                                   void* const* dst_ptrs, int32_t kernel, int32_t* path,
                                   int32_t* width);

/*
 * Work units of a tile: a single-row tile is split into 4096-byte units, a
 * multi-row tile into units of max(1, 4096 / (row_bytes + 256)) rows (256
 * bytes stand for each row's fixed work).  Each CTA of a copy kernel takes an
 * equal share of a program's units.  Returns 0 for NULL.
 */
int64_t reshard_tile_units(const reshard_tile_t* tile);

/*
 * Membership change (news.bpdata.com, section "Integracio es hibrid megoldas a
 * NeMo RL-ben": when GPUs join or leave at run time the communication group is
 * rebuilt, or shrunk/grown in place).  Derives a new plan from plan's layouts
 * (and in-place declaration) in which exactly the listed ranks are gone; rank
 * numbering is unchanged, so buffer tables keep M + N entries and a gone rank's
 * pointer may be NULL.  A gone source rank is never read: the regions it
 * served move to the remaining replicas of its box (rebalanced as at
 * creation); a gone destination rank is never written.  The derived plan's own
 * exclusions do not carry over: a rank that comes back is a call with a shorter
 * list (an empty one gives the full plan again).  An in-place alias that
 * involves a gone rank is dropped.  Errors: BAD_HANDLE, INVALID_ARG (rank out
 * of range, NULL list with a positive count), UNSUPPORTED (some destination
 * bytes have no remaining source rank), NO_MEMORY.
 */
reshard_status_t reshard_plan_exclude(reshard_plan_t plan, const int64_t* src_gone,
                                      int32_t n_src_gone, const int64_t* dst_gone,
                                      int32_t n_dst_gone, reshard_plan_t* out_plan);

/* Release a plan and its device tables.  Errors: BAD_HANDLE. */
reshard_status_t reshard_plan_destroy(reshard_plan_t plan);

/* Message of the last failed call on this thread ("" if none). */
const char* reshard_last_error(void);

/* Library version string. */
const char* reshard_version(void);

#ifdef __cplusplus
}
#endif

#endif /* RESHARD_H_ */
