/*
 * oracle.c -- plain, slow CPU reference of the DTensor-to-DTensor reshard.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: it exists so that tests, the smoke check and the CPU
 * baseline leg of the benchmark can compare the CUDA library against an
 * implementation that shares no code, header, table or helper with it.
 *
 * What it computes (the plain definition of the result, no planning):
 *   for every destination rank r, for every element of r's local shard,
 *   take its global index g, find the first source rank (flat order) whose
 *   shard box contains g, and copy the element's bytes from there.
 * Source: "Accelerating Reinforcement Learning Weight Refit with the Reshard
 * Collective" as summarised on news.bpdata.com (section "A megkozelites:
 * refit mint DTensor-to-DTensor reshard": a DTensor is a global shape, a
 * device mesh and placements; the refit is a reshard from the source layout
 * to the destination layout) and on techfeed.io (section "Reshard
 * Collective": the 8x8 worked example).
 *
 * Layout rule (resolve), pages silent -> DTensor's documented semantics:
 *   ranks are row-major coordinates on the mesh; mesh dims are applied in
 *   order (mesh dim 0 outermost); Shard(d) splits the CURRENT local extent n
 *   of tensor dim d into k = mesh[md] chunks of size ceil(n/k), chunk c is
 *   [min(c*ceil, n), min((c+1)*ceil, n)) (torch.chunk, short or empty
 *   trailing chunks); Replicate does not split.  A dim whose final local
 *   extent is zero reports offset = global extent (DTensor convention).
 *
 * Placement encoding used here (deliberately not the library's): one int32
 * per mesh dim, -1 = Replicate, d >= 0 = Shard(d).
 *
 * Local buffers are contiguous row-major arrays of the local shape.
 * Elements are opaque byte strings of elem_bytes (a bit copy: no dtype
 * arithmetic, NaN payloads and -0 survive).
 *
 * All functions return 0 on success and a negative code on failure:
 *   -1 invalid argument, -2 an element has no owning source shard,
 *   -3 out of host memory.
 *
 * Compile-time switch ORACLE_PLANT (tests only): plants one deliberate
 * mistake so that the test suite can show that its pins catch it.  It is
 * never defined in the normal build.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifndef ORACLE_PLANT
#define ORACLE_PLANT 0
#endif

#define ORACLE_MAX_NDIM 8

static int check_layout(int32_t ndim, const int64_t* gshape, int32_t mesh_ndim,
                        const int64_t* mesh, const int32_t* shard_dim) {
  if (ndim < 1 || ndim > ORACLE_MAX_NDIM || mesh_ndim < 1 || mesh_ndim > ORACLE_MAX_NDIM)
    return -1;
  for (int32_t d = 0; d < ndim; ++d)
    if (gshape[d] < 0) return -1;
  for (int32_t m = 0; m < mesh_ndim; ++m) {
    if (mesh[m] < 1) return -1;
    if (shard_dim[m] < -1 || shard_dim[m] >= ndim) return -1;
  }
  return 0;
}

static int64_t mesh_ranks(int32_t mesh_ndim, const int64_t* mesh) {
  int64_t n = 1;
  for (int32_t m = 0; m < mesh_ndim; ++m) n *= mesh[m];
  return n;
}

/* Local box (global offset + local shape) of one flat rank. */
int oracle_resolve(int32_t ndim, const int64_t* gshape, int32_t mesh_ndim, const int64_t* mesh,
                   const int32_t* shard_dim, int64_t rank, int64_t* offset, int64_t* shape) {
  if (check_layout(ndim, gshape, mesh_ndim, mesh, shard_dim)) return -1;
  int64_t nranks = mesh_ranks(mesh_ndim, mesh);
  if (rank < 0 || rank >= nranks) return -1;

  /* row-major coordinates of the rank on the mesh */
  int64_t coord[ORACLE_MAX_NDIM];
  int64_t rest = rank;
  for (int32_t m = mesh_ndim - 1; m >= 0; --m) {
    coord[m] = rest % mesh[m];
    rest /= mesh[m];
  }

  int sharded[ORACLE_MAX_NDIM];
  for (int32_t d = 0; d < ndim; ++d) {
    offset[d] = 0;
    shape[d] = gshape[d];
    sharded[d] = 0;
  }
#if ORACLE_PLANT == 5
  /* planted mistake: innermost mesh dim applied first */
  for (int32_t m = mesh_ndim - 1; m >= 0; --m) {
#else
  for (int32_t m = 0; m < mesh_ndim; ++m) {
#endif
    int32_t d = shard_dim[m];
    if (d < 0) continue; /* Replicate */
    int64_t n = shape[d];
    int64_t k = mesh[m];
#if ORACLE_PLANT == 1
    int64_t chunk = n / k; /* planted mistake: floor instead of ceil */
    if (chunk == 0) chunk = 1;
#else
    int64_t chunk = (n + k - 1) / k;
#endif
    int64_t lo = coord[m] * chunk;
    if (lo > n) lo = n;
    int64_t hi = lo + chunk;
    if (hi > n) hi = n;
#if ORACLE_PLANT == 7
    offset[d] = lo; /* planted mistake: outer split's offset dropped */
#else
    offset[d] += lo;
#endif
    shape[d] = hi - lo;
    sharded[d] = 1;
  }
#if ORACLE_PLANT != 6 /* planted mistake 6: empty-shard offset convention skipped */
  for (int32_t d = 0; d < ndim; ++d)
    if (sharded[d] && shape[d] == 0) offset[d] = gshape[d];
#endif
  (void)sharded;
  return 0;
}

static int64_t volume(int32_t ndim, const int64_t* shape) {
  int64_t v = 1;
  for (int32_t d = 0; d < ndim; ++d) v *= shape[d];
  return v;
}

/* Does box (off, shp) contain global index g? */
static int contains(int32_t ndim, const int64_t* off, const int64_t* shp, const int64_t* g) {
  for (int32_t d = 0; d < ndim; ++d) {
#if ORACLE_PLANT == 4
    if (g[d] < off[d] || g[d] > off[d] + shp[d]) return 0; /* planted: closed upper bound */
#else
    if (g[d] < off[d] || g[d] >= off[d] + shp[d]) return 0;
#endif
  }
  return 1;
}

/* Row-major linear index of multi-index i in a buffer of shape shp. */
static int64_t linear(int32_t ndim, const int64_t* i, const int64_t* shp) {
  int64_t lin = 0;
#if ORACLE_PLANT == 2
  /* planted mistake: column-major local layout */
  for (int32_t d = ndim - 1; d >= 0; --d) lin = lin * shp[d] + i[d];
#else
  for (int32_t d = 0; d < ndim; ++d) lin = lin * shp[d] + i[d];
#endif
  return lin;
}

typedef struct {
  int32_t ndim;
  int64_t nsrc;
  int64_t* off; /* [nsrc][ndim] */
  int64_t* shp; /* [nsrc][ndim] */
} src_boxes;

static int load_src_boxes(src_boxes* sb, int32_t ndim, const int64_t* gshape, int32_t mesh_ndim,
                          const int64_t* mesh, const int32_t* shard_dim) {
  sb->ndim = ndim;
  sb->nsrc = mesh_ranks(mesh_ndim, mesh);
  sb->off = (int64_t*)malloc(sizeof(int64_t) * (size_t)(sb->nsrc * ndim));
  sb->shp = (int64_t*)malloc(sizeof(int64_t) * (size_t)(sb->nsrc * ndim));
  if (!sb->off || !sb->shp) {
    free(sb->off);
    free(sb->shp);
    return -3;
  }
  for (int64_t s = 0; s < sb->nsrc; ++s) {
    int rc = oracle_resolve(ndim, gshape, mesh_ndim, mesh, shard_dim, s, sb->off + s * ndim,
                            sb->shp + s * ndim);
    if (rc) {
      free(sb->off);
      free(sb->shp);
      return rc;
    }
  }
  return 0;
}

static void free_src_boxes(src_boxes* sb) {
  free(sb->off);
  free(sb->shp);
}

/* First source rank (flat order) whose box holds global index g, or -1. */
static int64_t owner_of(const src_boxes* sb, const int64_t* g) {
  for (int64_t s = 0; s < sb->nsrc; ++s) {
    const int64_t* shp = sb->shp + s * sb->ndim;
    if (volume(sb->ndim, shp) == 0) continue;
    if (contains(sb->ndim, sb->off + s * sb->ndim, shp, g)) return s;
  }
  return -1;
}

/*
 * Elements [e_begin, e_end) (row-major linear indices) of destination rank r,
 * written to out (which holds the whole local shard of r).
 */
static int fill_rank(const src_boxes* sb, int32_t ndim, const int64_t* gshape, int64_t elem_bytes,
                     int32_t dst_mesh_ndim, const int64_t* dst_mesh, const int32_t* dst_shard_dim,
                     const void* const* src_bufs, int64_t r, int64_t e_begin, int64_t e_end,
                     unsigned char* out) {
  int64_t doff[ORACLE_MAX_NDIM], dshp[ORACLE_MAX_NDIM];
  oracle_resolve(ndim, gshape, dst_mesh_ndim, dst_mesh, dst_shard_dim, r, doff, dshp);
  int64_t n = volume(ndim, dshp);
  if (e_begin < 0 || e_end > n || e_begin > e_end) return -1;
  int64_t i[ORACLE_MAX_NDIM], g[ORACLE_MAX_NDIM], j[ORACLE_MAX_NDIM];
  /* local multi-index of element e_begin */
  int64_t rest = e_begin;
#if ORACLE_PLANT == 8
  /* planted mistake: start index unravelled with the first dim fastest */
  for (int32_t d = 0; d < ndim; ++d) {
#else
  for (int32_t d = ndim - 1; d >= 0; --d) {
#endif
    i[d] = dshp[d] ? rest % dshp[d] : 0;
#if ORACLE_PLANT != 9 /* planted mistake 9: the carry into the outer dims is dropped */
    rest = dshp[d] ? rest / dshp[d] : 0;
#endif
  }
  for (int64_t e = e_begin; e < e_end; ++e) {
    /* e is the row-major linear index of local multi-index i */
    for (int32_t d = 0; d < ndim; ++d) g[d] = doff[d] + i[d];
    int64_t s = owner_of(sb, g);
    if (s < 0) return -2;
    const int64_t* soff = sb->off + s * ndim;
    const int64_t* sshp = sb->shp + s * ndim;
    for (int32_t d = 0; d < ndim; ++d) j[d] = g[d] - soff[d];
    const unsigned char* in = (const unsigned char*)src_bufs[s];
    memcpy(out + linear(ndim, i, dshp) * elem_bytes, in + linear(ndim, j, sshp) * elem_bytes,
           (size_t)elem_bytes);
    /* advance the local multi-index (odometer, last dim fastest) */
    for (int32_t d = ndim - 1; d >= 0; --d) {
      if (++i[d] < dshp[d]) break;
      i[d] = 0;
    }
  }
  return 0;
}

/*
 * Fill destination ranks [dst_begin, dst_end) of the destination layout from
 * the source shards.  src_bufs[s] is source rank s's local buffer (may be NULL
 * for an empty shard), dst_bufs[r - dst_begin] is destination rank r's.
 */
int oracle_reshard(int32_t ndim, const int64_t* gshape, int64_t elem_bytes,
                   int32_t src_mesh_ndim, const int64_t* src_mesh, const int32_t* src_shard_dim,
                   int32_t dst_mesh_ndim, const int64_t* dst_mesh, const int32_t* dst_shard_dim,
                   const void* const* src_bufs, void* const* dst_bufs, int64_t dst_begin,
                   int64_t dst_end) {
  if (elem_bytes < 1) return -1;
  if (check_layout(ndim, gshape, dst_mesh_ndim, dst_mesh, dst_shard_dim)) return -1;
  int64_t ndst = mesh_ranks(dst_mesh_ndim, dst_mesh);
  if (dst_begin < 0 || dst_end > ndst || dst_begin > dst_end) return -1;

  src_boxes sb;
  int rc = load_src_boxes(&sb, ndim, gshape, src_mesh_ndim, src_mesh, src_shard_dim);
  if (rc) return rc;
  for (int64_t r = dst_begin; r < dst_end && rc == 0; ++r) {
    int64_t doff[ORACLE_MAX_NDIM], dshp[ORACLE_MAX_NDIM];
    oracle_resolve(ndim, gshape, dst_mesh_ndim, dst_mesh, dst_shard_dim, r, doff, dshp);
    rc = fill_rank(&sb, ndim, gshape, elem_bytes, dst_mesh_ndim, dst_mesh, dst_shard_dim,
                   src_bufs, r, 0, volume(ndim, dshp), (unsigned char*)dst_bufs[r - dst_begin]);
  }
  free_src_boxes(&sb);
  return rc;
}

/*
 * The same definition restricted to elements [e_begin, e_end) of one
 * destination rank (dst_buf holds that rank's whole local shard).  Used to
 * time the oracle on a bounded part of a large workload.
 */
int oracle_reshard_elems(int32_t ndim, const int64_t* gshape, int64_t elem_bytes,
                         int32_t src_mesh_ndim, const int64_t* src_mesh,
                         const int32_t* src_shard_dim, int32_t dst_mesh_ndim,
                         const int64_t* dst_mesh, const int32_t* dst_shard_dim,
                         const void* const* src_bufs, void* dst_buf, int64_t dst_rank,
                         int64_t e_begin, int64_t e_end) {
  if (elem_bytes < 1) return -1;
  if (check_layout(ndim, gshape, dst_mesh_ndim, dst_mesh, dst_shard_dim)) return -1;
  if (dst_rank < 0 || dst_rank >= mesh_ranks(dst_mesh_ndim, dst_mesh)) return -1;
  src_boxes sb;
  int rc = load_src_boxes(&sb, ndim, gshape, src_mesh_ndim, src_mesh, src_shard_dim);
  if (rc) return rc;
  rc = fill_rank(&sb, ndim, gshape, elem_bytes, dst_mesh_ndim, dst_mesh, dst_shard_dim, src_bufs,
                 dst_rank, e_begin, e_end, (unsigned char*)dst_buf);
  free_src_boxes(&sb);
  return rc;
}

/*
 * One element at a time: which source rank and which element of its local
 * buffer (row-major linear index) supply element dst_linear of destination
 * rank dst_rank.  Used to check outputs too large for oracle_reshard.
 */
int oracle_source_of(int32_t ndim, const int64_t* gshape, int32_t src_mesh_ndim,
                     const int64_t* src_mesh, const int32_t* src_shard_dim, int32_t dst_mesh_ndim,
                     const int64_t* dst_mesh, const int32_t* dst_shard_dim, int64_t dst_rank,
                     int64_t dst_linear, int64_t* src_rank, int64_t* src_linear) {
  if (check_layout(ndim, gshape, dst_mesh_ndim, dst_mesh, dst_shard_dim)) return -1;
  if (dst_rank < 0 || dst_rank >= mesh_ranks(dst_mesh_ndim, dst_mesh)) return -1;
  int64_t doff[ORACLE_MAX_NDIM], dshp[ORACLE_MAX_NDIM];
  oracle_resolve(ndim, gshape, dst_mesh_ndim, dst_mesh, dst_shard_dim, dst_rank, doff, dshp);
  if (dst_linear < 0 || dst_linear >= volume(ndim, dshp)) return -1;

  /* unravel the local linear index (row-major) */
  int64_t i[ORACLE_MAX_NDIM], g[ORACLE_MAX_NDIM], j[ORACLE_MAX_NDIM];
  int64_t rest = dst_linear;
  for (int32_t d = ndim - 1; d >= 0; --d) {
    i[d] = rest % dshp[d];
    rest /= dshp[d];
  }
  for (int32_t d = 0; d < ndim; ++d) g[d] = doff[d] + i[d];

  src_boxes sb;
  int rc = load_src_boxes(&sb, ndim, gshape, src_mesh_ndim, src_mesh, src_shard_dim);
  if (rc) return rc;
  int64_t s = owner_of(&sb, g);
  if (s < 0) {
    free_src_boxes(&sb);
    return -2;
  }
  for (int32_t d = 0; d < ndim; ++d) j[d] = g[d] - sb.off[s * ndim + d];
  *src_rank = s;
  *src_linear = linear(ndim, j, sb.shp + s * ndim);
  free_src_boxes(&sb);
  return 0;
}

/*
 * The conventional path's intermediate: the full global tensor, assembled
 * from the first replica of every source region (all-gather), as a plain
 * per-element loop over the global index space.
 */
int oracle_gather_full(int32_t ndim, const int64_t* gshape, int64_t elem_bytes,
                       int32_t src_mesh_ndim, const int64_t* src_mesh, const int32_t* src_shard_dim,
                       const void* const* src_bufs, void* full) {
  if (elem_bytes < 1) return -1;
  src_boxes sb;
  int rc = load_src_boxes(&sb, ndim, gshape, src_mesh_ndim, src_mesh, src_shard_dim);
  if (rc) return rc;
  int64_t n = volume(ndim, gshape);
  int64_t g[ORACLE_MAX_NDIM], j[ORACLE_MAX_NDIM];
  for (int32_t d = 0; d < ndim; ++d) g[d] = 0;
  unsigned char* out = (unsigned char*)full;
  for (int64_t e = 0; e < n; ++e) {
    int64_t s = owner_of(&sb, g);
    if (s < 0) {
      free_src_boxes(&sb);
      return -2;
    }
    for (int32_t d = 0; d < ndim; ++d) j[d] = g[d] - sb.off[s * ndim + d];
    memcpy(out + e * elem_bytes,
           (const unsigned char*)src_bufs[s] + linear(ndim, j, sb.shp + s * ndim) * elem_bytes,
           (size_t)elem_bytes);
    for (int32_t d = ndim - 1; d >= 0; --d) {
      if (++g[d] < gshape[d]) break;
      g[d] = 0;
    }
  }
  free_src_boxes(&sb);
  return 0;
}
