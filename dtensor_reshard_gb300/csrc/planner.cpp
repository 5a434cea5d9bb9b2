// planner.cpp -- host planner and C ABI of libreshard.so.
//
// The planner turns two DTensor layouts of one global tensor into copy
// programs for the CUDA kernels:
//   1. resolve every rank's box (global offset + local shape);
//   2. group ranks holding identical boxes into classes (replicas);
//   3. intersect every destination class with every source class;
//   4. pick one source replica per region, largest region first, onto the
//      replica with the fewest bytes read so far (ties: lowest rank);
//   5. express each region in both local layouts, collapse dims that are
//      contiguous in both, and cut it into tiles;
//   6. attach the destination replicas of the region's class as one fan-out
//      group and sort the tiles by destination.
// Steps 3-4 follow the Reshard collective write-ups (news.bpdata.com, section
// "A Reshard kollektiv kommunikacio": exact source/destination intersections
// first, each contribution sent once, replicas assemble locally; techfeed.io,
// section on NVIDIA's implementation: incoming data spread as evenly as
// possible across replicas).
#include <cuda_runtime.h>

#include <algorithm>
#include <chrono>
#include <climits>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <new>
#include <unordered_set>

#include "internal.h"

namespace rs {
namespace {

constexpr uint64_t kPlanMagic = 0x5245534841524431ull;  // "RESHARD1"

thread_local std::string g_last_error;

std::mutex g_registry_mu;
std::unordered_set<const reshard_plan_s*>& registry() {
  static std::unordered_set<const reshard_plan_s*> r;
  return r;
}

bool live(const reshard_plan_s* p) {
  if (!p) return false;
  std::lock_guard<std::mutex> lk(g_registry_mu);
  return registry().count(p) != 0;
}

int elem_size(int32_t dtype) {
  switch (dtype) {
    case RESHARD_U8: return 1;
    case RESHARD_BF16:
    case RESHARD_FP16: return 2;
    case RESHARD_FP32:
    case RESHARD_I32: return 4;
    case RESHARD_FP64:
    case RESHARD_I64: return 8;
    default: return 0;
  }
}

}  // namespace

// ---------------------------------------------------------------- step 1: resolve
// Shard(d) on a mesh dim of size k splits the current local extent n of dim d
// into torch.chunk pieces of ceil(n/k); mesh dims apply in order.
void resolve_rank(int32_t nd, const int64_t* gshape, const Layout& L, int64_t rank, Box* b) {
  int64_t coord[RESHARD_MAX_MESH_NDIM];
  int64_t rest = rank;
  for (int m = L.mesh_ndim - 1; m >= 0; --m) {
    coord[m] = rest % L.mesh[m];
    rest /= L.mesh[m];
  }
  bool sharded[RESHARD_MAX_TENSOR_NDIM] = {};
  for (int d = 0; d < nd; ++d) {
    b->off[d] = 0;
    b->shp[d] = gshape[d];
  }
  for (int m = 0; m < L.mesh_ndim; ++m) {
    if (L.pl[m].kind != RESHARD_SHARD) continue;
    const int d = L.pl[m].dim;
    const int64_t n = b->shp[d];
    const int64_t piece = (n + L.mesh[m] - 1) / L.mesh[m];
    const int64_t lo = std::min(coord[m] * piece, n);
    const int64_t hi = std::min(lo + piece, n);
    b->off[d] += lo;
    b->shp[d] = hi - lo;
    sharded[d] = true;
  }
  for (int d = 0; d < nd; ++d)
    if (sharded[d] && b->shp[d] == 0) b->off[d] = gshape[d];
}

int64_t box_volume(int32_t nd, const Box& b) {
  int64_t v = 1;
  for (int d = 0; d < nd; ++d) v *= b.shp[d];
  return v;
}

// ---------------------------------------------------------------- step 2: classes
std::vector<Class> classes_of(int32_t nd, const Layout& L, const std::vector<uint8_t>& gone) {
  std::vector<Class> out;
  std::map<std::vector<int64_t>, size_t> index;
  for (int64_t r = 0; r < L.nranks; ++r) {
    if (!gone.empty() && gone[size_t(r)]) continue;
    const Box& b = L.box[r];
    const int64_t vol = box_volume(nd, b);
    if (vol == 0) continue;
    std::vector<int64_t> key(b.off, b.off + nd);
    key.insert(key.end(), b.shp, b.shp + nd);
    auto it = index.find(key);
    if (it == index.end()) {
      index.emplace(key, out.size());
      Class c;
      c.box = b;
      c.volume = vol;
      c.ranks.push_back(r);
      out.push_back(c);
    } else {
      out[it->second].ranks.push_back(r);
    }
  }
  return out;
}

// ---------------------------------------------------------------- step 5: tiles

void row_major_strides(int32_t nd, const int64_t* shp, int64_t* st) {
  int64_t s = 1;
  for (int d = nd - 1; d >= 0; --d) {
    st[d] = s;
    s *= shp[d];
  }
}

// Emit the tiles copying a box of extents e[nd] (elements) that starts at
// element src_base / dst_base of buffers with strides sst / dst (elements).
void emit_box(Program& P, uint16_t src_buf, uint16_t group, int32_t nd, const int64_t* e,
              int64_t src_base, const int64_t* sst, int64_t dst_base, const int64_t* dstr,
              int64_t eb, int64_t fanout) {
  std::vector<Dim> dims;
  for (int d = 0; d < nd; ++d) {
    if (e[d] == 0) return;
    if (e[d] > 1) dims.push_back({e[d], sst[d], dstr[d]});
  }
  // merge neighbours that are contiguous in both layouts
  std::vector<Dim> m;
  for (const Dim& d : dims) {
    if (!m.empty() && m.back().ss == d.e * d.ss && m.back().ds == d.e * d.ds) {
      m.back() = {m.back().e * d.e, d.ss, d.ds};
    } else {
      m.push_back(d);
    }
  }
  int64_t row_elems = 1;
  if (!m.empty() && m.back().ss == 1 && m.back().ds == 1) {
    row_elems = m.back().e;
    m.pop_back();
  }
  const int64_t row_bytes = row_elems * eb;
  // A single row, or rows longer than kRunSplitBytes, become run tiles (one
  // per row, cut into pieces of at most kMaxRunBytes).
  auto emit_run = [&](int64_t sbyte, int64_t dbyte) {
    for (int64_t o = 0; o < row_bytes; o += kMaxRunBytes) {
      reshard_tile_t t = {};
      t.src_off = sbyte + o;
      t.dst_off = dbyte + o;
      t.row_bytes = uint32_t(std::min(kMaxRunBytes, row_bytes - o));
      t.nrows = t.nplanes = 1;
      t.src_buf = src_buf;
      t.dst_group = group;
      P.tiles.push_back(t);
    }
  };
  auto emit_rows = [&](int64_t sb, int64_t db, int64_t nplanes, int64_t sps, int64_t dps,
                       int64_t nrows, int64_t srs, int64_t drs) {
    if (nplanes * nrows == 1 || row_bytes > kRunSplitBytes) {
      for (int64_t p = 0; p < nplanes; ++p)
        for (int64_t r = 0; r < nrows; ++r)
          emit_run((sb + p * sps + r * srs) * eb, (db + p * dps + r * drs) * eb);
      return;
    }
    // keep nrows * nplanes of one tile below 2^30: slice planes, then rows
    const int64_t kMaxRows = int64_t(1) << 30;
    const int64_t pstep = std::max<int64_t>(1, kMaxRows / nrows);
    // rows that are a column band of wider destination rows: cut into blocks
    int64_t rstep = kMaxRows;
    if (kGatherBlockBytes > 0 && fanout >= kGatherBlockFanout && nplanes == 1 &&
        drs * eb > row_bytes)
      rstep = std::max<int64_t>(int64_t(rows_per_unit(uint32_t(row_bytes))),
                                (kGatherBlockBytes + row_bytes - 1) / row_bytes);
    for (int64_t p0 = 0; p0 < nplanes; p0 += pstep) {
      const int64_t np = std::min(nplanes - p0, pstep);
      for (int64_t r0 = 0; r0 < nrows; r0 += rstep) {
        const int64_t nr = std::min(nrows - r0, rstep);
        reshard_tile_t t = {};
        t.src_off = (sb + p0 * sps + r0 * srs) * eb;
        t.dst_off = (db + p0 * dps + r0 * drs) * eb;
        t.row_bytes = uint32_t(row_bytes);
        t.nrows = uint32_t(nr);
        t.nplanes = uint32_t(np);
        if (t.nrows > 1) {
          t.src_row_stride = srs * eb;
          t.dst_row_stride = drs * eb;
        }
        if (t.nplanes > 1) {
          t.src_plane_stride = sps * eb;
          t.dst_plane_stride = dps * eb;
        }
        t.src_buf = src_buf;
        t.dst_group = group;
        P.tiles.push_back(t);
      }
    }
  };
  const size_t k = m.size();
  if (k == 0) {
    emit_rows(src_base, dst_base, 1, 0, 0, 1, 0, 0);
  } else if (k == 1) {
    emit_rows(src_base, dst_base, 1, 0, 0, m[0].e, m[0].ss, m[0].ds);
  } else {
    // outer dims beyond two become a loop of 2-level tiles
    const Dim& pl = m[k - 2];
    const Dim& rw = m[k - 1];
    std::vector<int64_t> idx(k - 2, 0);
    while (true) {
      int64_t sb = src_base, db = dst_base;
      for (size_t i = 0; i + 2 < k; ++i) {
        sb += idx[i] * m[i].ss;
        db += idx[i] * m[i].ds;
      }
      emit_rows(sb, db, pl.e, pl.ss, pl.ds, rw.e, rw.ss, rw.ds);
      int64_t i = int64_t(k) - 3;
      for (; i >= 0; --i) {
        if (++idx[i] < m[i].e) break;
        idx[i] = 0;
      }
      if (i < 0) break;
    }
  }
}

void finish_program(Program& P) {
  // sort by destination (first buffer of the group, then offset)
  std::stable_sort(P.tiles.begin(), P.tiles.end(),
                   [&](const reshard_tile_t& a, const reshard_tile_t& b) {
                     const uint16_t ba = P.gbuf[P.goff[a.dst_group]];
                     const uint16_t bb = P.gbuf[P.goff[b.dst_group]];
                     if (ba != bb) return ba < bb;
                     if (a.dst_off != b.dst_off) return a.dst_off < b.dst_off;
                     return a.dst_group < b.dst_group;
                   });
  P.prefix.assign(P.tiles.size() + 1, 0);
  for (size_t i = 0; i < P.tiles.size(); ++i) {
    const reshard_tile_t& t = P.tiles[i];
    P.prefix[i + 1] = P.prefix[i] + tile_units(t);
    P.align_bits |= uint64_t(t.src_off) | uint64_t(t.dst_off) | t.row_bytes |
                    uint64_t(t.src_row_stride) | uint64_t(t.dst_row_stride) |
                    uint64_t(t.src_plane_stride) | uint64_t(t.dst_plane_stride);
    if (t.nplanes > 1) P.has_planes = true;
    const int64_t bytes = int64_t(t.row_bytes) * t.nrows * t.nplanes;
    P.tile_bytes += bytes;
    P.write_bytes += bytes * int64_t(P.goff[t.dst_group + 1] - P.goff[t.dst_group]);
    if (t.row_bytes >= 512) P.long_row_bytes += bytes;
    if (t.row_bytes >= 8192) P.wide_row_bytes += bytes;
    if (t.row_bytes < kNarrowRow) P.narrow_row_bytes += bytes;
  }
  for (size_t g = 0; g + 1 < P.goff.size(); ++g)
    P.max_fanout = std::max<int>(P.max_fanout, int(P.goff[g + 1] - P.goff[g]));
}

int64_t tile_bytes(const reshard_tile_t& t) {
  return int64_t(t.row_bytes) * t.nrows * t.nplanes;
}

namespace {

// ---------------------------------------------------------------- validation
reshard_status_t read_layout(const char* side, int32_t nd, const reshard_mesh_t* mesh,
                             const reshard_placement_t* pl, Layout* L) {
  if (!mesh || !pl) return fail(RESHARD_ERR_INVALID_ARG, std::string(side) + ": null mesh or placements");
  if (mesh->ndim < 1 || mesh->ndim > RESHARD_MAX_MESH_NDIM)
    return fail(RESHARD_ERR_UNSUPPORTED, std::string(side) + ": mesh ndim must be 1..4");
  L->mesh_ndim = mesh->ndim;
  L->nranks = 1;
  for (int m = 0; m < mesh->ndim; ++m) {
    if (mesh->shape[m] < 1)
      return fail(RESHARD_ERR_INVALID_ARG, std::string(side) + ": mesh sizes must be >= 1");
    if (mesh->shape[m] > RESHARD_MAX_RANKS || L->nranks * mesh->shape[m] > RESHARD_MAX_RANKS)
      return fail(RESHARD_ERR_UNSUPPORTED, std::string(side) + ": too many ranks");
    L->mesh[m] = mesh->shape[m];
    L->nranks *= mesh->shape[m];
    if (pl[m].kind == RESHARD_SHARD) {
      if (pl[m].dim < 0 || pl[m].dim >= nd)
        return fail(RESHARD_ERR_INVALID_ARG, std::string(side) + ": Shard dim out of range");
    } else if (pl[m].kind != RESHARD_REPLICATE) {
      return fail(RESHARD_ERR_UNSUPPORTED,
                  std::string(side) + ": only Shard and Replicate placements are supported");
    }
    L->pl[m] = pl[m];
    if (L->pl[m].kind == RESHARD_REPLICATE) L->pl[m].dim = 0;
  }
  return RESHARD_OK;
}

// A region seen from one side as `rows` rows of `width` bytes at `stride`
// bytes apart starting at byte `base` (outer dims must collapse to one stride).
struct RowView {
  bool ok = false;
  int64_t base = 0, stride = 0, rows = 1, width = 0;
};

RowView row_view(int32_t nd, const int64_t* lo, const int64_t* ext, const Box& side, int64_t eb) {
  RowView v;
  int64_t st[RESHARD_MAX_TENSOR_NDIM];
  row_major_strides(nd, side.shp, st);
  v.width = ext[nd - 1] * eb;
  for (int k = 0; k < nd; ++k) v.base += (lo[k] - side.off[k]) * st[k] * eb;
  std::vector<Dim> m;
  for (int k = 0; k + 1 < nd; ++k) {
    if (ext[k] <= 1) continue;
    const Dim d = {ext[k], st[k], 0};
    if (!m.empty() && m.back().ss == d.e * d.ss) m.back() = {m.back().e * d.e, d.ss, 0};
    else m.push_back(d);
  }
  if (m.size() > 1) return v;
  v.rows = m.empty() ? 1 : m[0].e;
  v.stride = m.empty() ? 0 : m[0].ss * eb;
  v.ok = true;
  return v;
}

// A region's bytes on one side as planes x rows x width: rows along tensor dim
// nd - 2, planes over the dims before it, which must collapse into one level.
// For regions whose rows do not collapse into one level (a 3-D piece of a
// shard whose middle dim is cut as well).
struct PlaneView {
  bool ok = false;
  int64_t base = 0, pstride = 0, planes = 1, stride = 0, rows = 1, width = 0;
};

PlaneView plane_view(int32_t nd, const int64_t* lo, const int64_t* ext, const Box& side,
                     int64_t eb) {
  PlaneView v;
  if (nd < 3) return v;
  int64_t st[RESHARD_MAX_TENSOR_NDIM];
  row_major_strides(nd, side.shp, st);
  v.width = ext[nd - 1] * eb;
  for (int k = 0; k < nd; ++k) v.base += (lo[k] - side.off[k]) * st[k] * eb;
  v.rows = ext[nd - 2];
  v.stride = st[nd - 2] * eb;
  std::vector<Dim> m;
  for (int k = 0; k + 2 < nd; ++k) {
    if (ext[k] <= 1) continue;
    const Dim d = {ext[k], st[k], 0};
    if (!m.empty() && m.back().ss == d.e * d.ss) m.back() = {m.back().e * d.e, d.ss, 0};
    else m.push_back(d);
  }
  if (m.size() > 1) return v;
  v.planes = m.empty() ? 1 : m[0].e;
  v.pstride = m.empty() ? 0 : m[0].ss * eb;
  v.ok = true;
  return v;
}

PlaneView as_planes(const RowView& r) {
  PlaneView v;
  v.ok = r.ok;
  v.base = r.base;
  v.stride = r.stride;
  v.rows = r.rows;
  v.width = r.width;
  return v;
}

reshard_status_t build_plan(reshard_plan_s* P) {
  const int32_t nd = P->ndim;
  const int64_t eb = P->elem_bytes;
  const int64_t M = P->src.nranks, N = P->dst.nranks;

  reshard_stats_t& S = P->stats;
  S.global_bytes = eb;
  for (int d = 0; d < nd; ++d) S.global_bytes *= P->gshape[d];
  S.n_src_ranks = M;
  S.n_dst_ranks = N;
  auto present = [](const std::vector<uint8_t>& gone, int64_t r) {
    return gone.empty() || !gone[size_t(r)];
  };
  for (int64_t r = 0; r < M; ++r)
    if (present(P->src_gone, r)) S.src_bytes += box_volume(nd, P->src.box[r]) * eb;
  for (int64_t r = 0; r < N; ++r)
    if (present(P->dst_gone, r)) S.dst_bytes += box_volume(nd, P->dst.box[r]) * eb;

  const std::vector<Class> sc = classes_of(nd, P->src, P->src_gone);
  const std::vector<Class> dc = classes_of(nd, P->dst, P->dst_gone);
  S.n_src_classes = int64_t(sc.size());
  S.n_dst_classes = int64_t(dc.size());

  // ---- step 3: intersections
  struct Region {
    size_t d, s;
    int64_t lo[RESHARD_MAX_TENSOR_NDIM], ext[RESHARD_MAX_TENSOR_NDIM];
    int64_t bytes;
    int64_t replica = -1;
  };
  std::vector<Region> regions;
  for (size_t di = 0; di < dc.size(); ++di) {
    for (size_t si = 0; si < sc.size(); ++si) {
      Region g;
      g.d = di;
      g.s = si;
      int64_t vol = 1;
      for (int d = 0; d < nd; ++d) {
        const int64_t lo = std::max(dc[di].box.off[d], sc[si].box.off[d]);
        const int64_t hi = std::min(dc[di].box.off[d] + dc[di].box.shp[d],
                                    sc[si].box.off[d] + sc[si].box.shp[d]);
        if (hi <= lo) {
          vol = 0;
          break;
        }
        g.lo[d] = lo;
        g.ext[d] = hi - lo;
        vol *= hi - lo;
      }
      if (vol == 0) continue;
      g.bytes = vol * eb;
      regions.push_back(g);
    }
  }
  S.n_regions = int64_t(regions.size());
  for (const Region& g : regions) S.region_bytes += g.bytes;
  if (!P->src_gone.empty()) {
    // with source ranks gone, every destination class must still be covered
    std::vector<int64_t> covered(dc.size(), 0);
    for (const Region& g : regions) covered[g.d] += g.bytes;
    for (size_t di = 0; di < dc.size(); ++di)
      if (covered[di] != dc[di].volume * eb)
        return fail(RESHARD_ERR_UNSUPPORTED,
                    "no remaining source rank holds part of destination rank " +
                        std::to_string(dc[di].ranks[0]));
  }

  // ---- step 4: replica pick, largest region first onto the least-loaded replica
  {
    std::vector<size_t> order(regions.size());
    for (size_t i = 0; i < order.size(); ++i) order[i] = i;
    std::stable_sort(order.begin(), order.end(),
                     [&](size_t a, size_t b) { return regions[a].bytes > regions[b].bytes; });
    std::vector<int64_t> load(size_t(M), 0);
    for (size_t i : order) {
      Region& g = regions[i];
      int64_t best = -1;
      for (int64_t r : sc[g.s].ranks)
        if (best < 0 || load[size_t(r)] < load[size_t(best)]) best = r;
      g.replica = best;
      load[size_t(best)] += g.bytes;
    }
    for (int64_t r = 0; r < M; ++r) S.max_replica_read_bytes = std::max(S.max_replica_read_bytes, load[size_t(r)]);
  }

  // ---- step 6 (groups first): destination groups
  const uint16_t scratch_buf = uint16_t(M + N);
  Program& PF = P->prog[RESHARD_PROGRAM_FANOUT];
  Program& PB = P->prog[RESHARD_PROGRAM_BOXCOPY];
  Program& PG = P->prog[RESHARD_PROGRAM_GATHER];
  Program& PS = P->prog[RESHARD_PROGRAM_SLICE];
  Program& PR = P->prog[RESHARD_PROGRAM_REPLICATE];
  for (Program* p : {&PF, &PB, &PG, &PS, &PR}) p->goff.push_back(0);
  for (size_t di = 0; di < dc.size(); ++di)
    S.max_fanout = std::max<int64_t>(S.max_fanout, int64_t(dc[di].ranks.size()));
  // FANOUT groups, one per distinct list of target ranks (a destination class,
  // minus the ranks that already hold the region in place), at most kMaxGroup each
  std::map<std::vector<int64_t>, std::vector<uint16_t>> group_ids;
  bool too_many_groups = false;
  auto fan_groups = [&](const std::vector<int64_t>& ranks) -> const std::vector<uint16_t>& {
    auto it = group_ids.find(ranks);
    if (it != group_ids.end()) return it->second;
    std::vector<uint16_t> ids;
    for (size_t a = 0; a < ranks.size(); a += kMaxGroup) {
      if (PF.goff.size() > 65535) too_many_groups = true;
      ids.push_back(uint16_t(PF.goff.size() - 1));
      for (size_t b = a; b < std::min(ranks.size(), a + size_t(kMaxGroup)); ++b)
        PF.gbuf.push_back(uint16_t(M + ranks[b]));
      PF.goff.push_back(uint32_t(PF.gbuf.size()));
    }
    return group_ids.emplace(ranks, ids).first->second;
  };
  // one group per destination rank (BOXCOPY and SLICE)
  for (Program* p : {&PB, &PS}) {
    for (int64_t r = 0; r < N; ++r) {
      p->gbuf.push_back(uint16_t(M + r));
      p->goff.push_back(uint32_t(p->gbuf.size()));
    }
  }
  PG.gbuf.push_back(scratch_buf);
  PG.goff.push_back(1);

  // ---- step 5a: transpose blocks for narrow innermost pieces (fan-out program)
  std::vector<char> consumed(regions.size(), 0);
  if (!P->inplace && nd >= 2) {
    struct Piece {
      size_t ri;
      PlaneView wide, narrow;
      int64_t col;
    };
    // Emits the blocks of one group; `gather` = narrow sources into one destination class.
    // Blocks stay inside one plane of `rows` wide rows (wide planes wide_pstride apart).
    auto emit_group = [&](std::vector<Piece>& ps, bool gather, int64_t planes, int64_t rows,
                          int64_t L, int64_t wide_base, int64_t wide_pstride,
                          const std::vector<uint16_t>& wide_ids) {
      std::sort(ps.begin(), ps.end(), [](const Piece& a, const Piece& b) { return a.col < b.col; });
      // narrow buffer (gather) or destination groups (scatter) of every piece, once
      std::vector<std::vector<uint16_t>> narrow_ids(ps.size());
      for (size_t i = 0; i < ps.size(); ++i) {
        const Region& g = regions[ps[i].ri];
        if (gather) narrow_ids[i].push_back(uint16_t(g.replica));
        else narrow_ids[i] = fan_groups(dc[g.d].ranks);
      }
      // rows per block: enough blocks to occupy the GPU, at most one shared-memory image
      int64_t nb = std::min<int64_t>(
          rows, std::max<int64_t>(1, std::min<int64_t>(kTransposeBlockBytes / L,
                                                       (planes * rows + kTransposeMinBlocks - 1) /
                                                           kTransposeMinBlocks)));
      // a multiple of the rows after which the narrow ranges are back at the same
      // address mod 16 (then the kernel keeps their granule plans from block to
      // block): of every piece when that cut costs at most a quarter of the block
      // (a scatter of 32 pieces of 4 bytes and one of 2: 152-row blocks, 0.148 ms;
      // 156 rows, the 2-byte piece moving, 0.168 ms), else of the most common
      // width whatever the cut (a gather of 42 pieces of 68 bytes: 0.090 ms with
      // 4-row blocks, 0.103 ms with 7)
      {
        auto multiple = [](int64_t w) {
          int64_t m = 16;
          while (w > 0 && w % 2 == 0 && m > 1) {
            w /= 2;
            m /= 2;
          }
          return m;  // 16 / gcd(16, w)
        };
        std::map<int64_t, int64_t> count;
        int64_t m_all = 1;
        for (const Piece& pc : ps) {
          ++count[pc.narrow.width];
          m_all = std::max(m_all, multiple(pc.narrow.width));  // powers of two: the lcm
        }
        int64_t common = 0, most = -1;
        for (const auto& kv : count)
          if (kv.second > most) {
            most = kv.second;
            common = kv.first;
          }
        if (nb >= m_all && 4 * (nb % m_all) <= nb) {
          nb -= nb % m_all;
        } else {
          const int64_t m = multiple(common);
          if (nb >= m) nb -= nb % m;
        }
      }
      for (uint16_t wid : wide_ids) {
        for (int64_t pl = 0; pl < planes; ++pl) {
          for (int64_t r0 = 0; r0 < rows; r0 += nb) {
            reshard_tblock_t blk = {};
            // same shape as the block before it (same wide side, rows and segments;
            // only the offsets move): the kernel keeps what it worked out for it
            if (r0 > 0 || pl > 0) {
              const int64_t prev_rows = r0 > 0 ? nb : std::min(nb, rows - (rows - 1) / nb * nb);
              if (std::min(nb, rows - r0) == prev_rows) {
                blk.flags = RESHARD_TBLOCK_SAME_SHAPE;
                // inside a plane its rows and narrow ranges also follow the previous ones
                if (r0 > 0) blk.flags |= RESHARD_TBLOCK_FOLLOWS;
              }
            }
            blk.wide_off = wide_base + pl * wide_pstride + r0 * L;
            blk.row_bytes = uint32_t(L);
            blk.nrows = uint32_t(std::min(nb, rows - r0));
            blk.seg_begin = uint32_t(PF.tsegs.size());
            blk.wide = wid;
            blk.direction = gather ? 0 : 1;
            for (size_t i = 0; i < ps.size(); ++i) {
              const Piece& pc = ps[i];
              for (uint16_t nid : narrow_ids[i]) {
                reshard_tseg_t sg = {};
                sg.narrow_off = pc.narrow.base + pl * pc.narrow.pstride + r0 * pc.narrow.width;
                sg.width = uint32_t(pc.narrow.width);
                sg.col = uint32_t(pc.col);
                sg.narrow = nid;
                PF.tsegs.push_back(sg);
              }
            }
            blk.seg_count = uint32_t(PF.tsegs.size()) - blk.seg_begin;
            PF.tblocks.push_back(blk);
          }
        }
      }
      for (const Piece& pc : ps) consumed[pc.ri] = 1;
    };
    // Checks a candidate group: same rows (and planes), narrow sides dense within a
    // plane, wide side covered exactly.  Rows that collapse into one level on both
    // sides are one plane; otherwise the group is tried as planes of rows.
    auto try_group = [&](const std::vector<size_t>& members, bool gather) {
      if (members.size() < 2 || members.size() > size_t(kTransposeMaxSegs)) return;
      for (size_t ri : members)
        if (consumed[ri]) return;
      std::vector<Piece> ps;
      int64_t planes = -1, rows = -1, L = -1, wps = -1, base = INT64_MAX;
      for (int as_plane_rows = 0; as_plane_rows < 2 && ps.size() != members.size();
           ++as_plane_rows) {
        ps.clear();
        planes = rows = L = wps = -1;
        base = INT64_MAX;
        for (size_t ri : members) {
          const Region& g = regions[ri];
          const Box& sb = P->src.box[size_t(g.replica)];
          const Box& db = dc[g.d].box;
          const PlaneView sv = as_plane_rows ? plane_view(nd, g.lo, g.ext, sb, eb)
                                             : as_planes(row_view(nd, g.lo, g.ext, sb, eb));
          const PlaneView dv = as_plane_rows ? plane_view(nd, g.lo, g.ext, db, eb)
                                             : as_planes(row_view(nd, g.lo, g.ext, db, eb));
          if (!sv.ok || !dv.ok) break;
          const PlaneView& wide = gather ? dv : sv;
          const PlaneView& narrow = gather ? sv : dv;
          if (narrow.width >= kTransposeMaxWidth) break;
          if (rows < 0) {
            planes = wide.planes;
            rows = wide.rows;
            L = wide.stride;
            wps = wide.pstride;
          }
          if (wide.rows != rows || rows < 2 || narrow.rows != rows) break;
          if (wide.planes != planes || narrow.planes != planes || wide.pstride != wps) break;
          if (narrow.stride != narrow.width) break;  // narrow side dense within a plane
          if (wide.stride != L) break;
          base = std::min(base, wide.base);
          ps.push_back({ri, wide, narrow, 0});
        }
      }
      if (ps.size() != members.size()) return;
      if (L <= 0 || L > kTransposeBlockBytes) return;
      int64_t covered = 0;
      for (Piece& pc : ps) {
        pc.col = pc.wide.base - base;
        if (pc.col < 0 || pc.col + pc.wide.width > L) return;
        covered += pc.wide.width;
      }
      if (covered != L) return;  // with disjoint regions: exact cover of every wide row
      // Measured on GB300 (uneven-stress tensors): regrouping pays when a gather
      // fans out to several destination replicas, or when the pieces are narrow
      // (at most 32 bytes) and numerous (a scatter of 45 pieces of 32 bytes: 0.250
      // -> 0.205 ms; of 47 pieces of 18 bytes: 0.059 -> 0.049 ms), or for gathers
      // of 16 or more pieces up to 128 bytes into wide rows short enough for four
      // of them per block (42 pieces of 68 bytes: 0.133 -> 0.113 ms; 55 of 72
      // bytes: 0.018 -> 0.014 ms), or for scatters of rows of at most 8 bytes (3
      // pieces of 2 bytes: 0.176 -> 0.125 ms).  With fewer pieces of longer rows (8
      // pieces of 4 bytes out of 32-byte rows: 0.15 -> 0.34 ms), wider scatters (68-byte
      // pieces: +0.008 ms) or gathers into rows of 9 KB (two rows per block:
      // +0.008 ms), per-piece copies are faster.
      int64_t max_w = 0;
      for (const Piece& pc : ps) max_w = std::max(max_w, pc.narrow.width);
      const bool fanned = gather && dc[regions[members[0]].d].ranks.size() >= 2;
      // a scatter of rows of at most 8 bytes (a de-interleave): the per-piece copies
      // read every source sector once per piece, the blocks once
      const bool tiny_scatter = !gather && L <= 8;
      const bool narrow_many = (max_w <= 32 && ps.size() >= 16) || tiny_scatter;
      const bool gather_wide = gather && max_w <= 128 && ps.size() >= 16 &&
                               4 * L <= kTransposeBlockBytes;
      if (!fanned && !narrow_many && !gather_wide) return;
      if (!gather) {
        size_t nsegs = 0;
        for (const Piece& pc : ps) {
          const size_t R = dc[regions[pc.ri].d].ranks.size();
          nsegs += (R + kMaxGroup - 1) / kMaxGroup;
        }
        if (nsegs > size_t(kTransposeMaxSegs)) return;
        size_t nptrs = 0;
        for (const Piece& pc : ps) nptrs += dc[regions[pc.ri].d].ranks.size();
        if (nptrs > size_t(kTransposeMaxReplicaPtrs)) return;
      }
      std::vector<uint16_t> wide_ids;
      if (gather) wide_ids = fan_groups(dc[regions[members[0]].d].ranks);
      else wide_ids.push_back(uint16_t(regions[members[0]].replica));
      emit_group(ps, gather, planes, rows, L, base, wps, wide_ids);
    };
    std::vector<std::vector<size_t>> into(dc.size()), outof(sc.size());
    for (size_t ri = 0; ri < regions.size(); ++ri) {
      into[regions[ri].d].push_back(ri);
      outof[regions[ri].s].push_back(ri);
    }
    // gather: all regions into one destination class
    for (size_t di = 0; di < dc.size(); ++di) try_group(into[di], true);
    // scatter: all regions out of one source class, read from one replica
    for (size_t si = 0; si < sc.size(); ++si) {
      std::vector<size_t> members;
      for (size_t ri : outof[si])
        if (!consumed[ri]) members.push_back(ri);
      if (members.size() < 2) continue;
      bool same = true;
      for (size_t ri : members) same = same && regions[ri].replica == regions[members[0]].replica;
      if (!same) {
        std::vector<int64_t> saved;
        for (size_t ri : members) saved.push_back(regions[ri].replica);
        for (size_t ri : members) regions[ri].replica = regions[members[0]].replica;
        try_group(members, false);
        if (!consumed[members[0]])
          for (size_t k = 0; k < members.size(); ++k) regions[members[k]].replica = saved[k];
      } else {
        try_group(members, false);
      }
    }
  }

  // ---- step 5b: tiles
  int64_t gst[RESHARD_MAX_TENSOR_NDIM];
  row_major_strides(nd, P->gshape, gst);
  // Region placement in its source replica and destination class (element offsets
  // and strides of both local layouts).
  struct Place {
    int64_t s0 = 0, d0 = 0;
    int64_t sst[RESHARD_MAX_TENSOR_NDIM] = {}, dst[RESHARD_MAX_TENSOR_NDIM] = {};
  };
  auto place_of = [&](const Region& g) {
    Place q;
    const Box& sb = P->src.box[size_t(g.replica)];
    const Box& db = dc[g.d].box;
    row_major_strides(nd, sb.shp, q.sst);
    row_major_strides(nd, db.shp, q.dst);
    for (int d = 0; d < nd; ++d) {
      q.s0 += (g.lo[d] - sb.off[d]) * q.sst[d];
      q.d0 += (g.lo[d] - db.off[d]) * q.dst[d];
    }
    return q;
  };
  // Destination classes assembled in one replica (their first rank) and then
  // replicated: many replicas, several regions meeting in each shard (a single
  // region would be copied twice for nothing), every region on per-piece tiles
  // (no transpose block), and tiles that would take the register realigning kernel (off the
  // 16-byte grid, mostly rows of 512 bytes and more, not mostly rows of 8 KiB
  // in a class large enough for the staged kernel).  The pages' two-stage
  // transfer reads the same way: one copy crosses once, then is replicated
  // where it landed.
  std::vector<int64_t> assemble_at(dc.size(), -1);
  if (!P->inplace) {
    std::vector<std::vector<size_t>> of_class(dc.size());
    for (size_t ri = 0; ri < regions.size(); ++ri) of_class[regions[ri].d].push_back(ri);
    for (size_t di = 0; di < dc.size(); ++di) {
      if (int64_t(dc[di].ranks.size()) < kAssembleFanout || of_class[di].size() < 2) continue;
      bool blocked = false;
      for (size_t ri : of_class[di]) blocked = blocked || consumed[ri];
      if (blocked) continue;
      Program T;
      T.goff = {0, 1};
      T.gbuf = {0};
      for (size_t ri : of_class[di]) {
        const Region& g = regions[ri];
        const Place q = place_of(g);
        emit_box(T, 0, 0, nd, g.ext, q.s0, q.sst, q.d0, q.dst, eb);
      }
      finish_program(T);
      const bool aligned = (T.align_bits & 15u) == 0;
      const bool long_rows = 2 * T.long_row_bytes >= T.tile_bytes;
      const bool staged = 2 * T.wide_row_bytes >= T.tile_bytes && T.tile_bytes >= (int64_t(48) << 20);
      if (!aligned && long_rows && !staged) assemble_at[di] = dc[di].ranks[0];
    }
  }
  for (size_t ri = 0; ri < regions.size(); ++ri) {
    const Region& g = regions[ri];
    // destination ranks that still need the region (in-place plans drop the
    // rank whose buffer already holds a source replica of it)
    std::vector<int64_t> targets;
    for (int64_t r : dc[g.d].ranks) {
      bool in_place = false;
      if (P->inplace)
        for (int64_t s : sc[g.s].ranks)
          if (P->alias_dst[size_t(s)] == r) in_place = true;
      if (!in_place) targets.push_back(r);
    }
    S.inplace_bytes += g.bytes * int64_t(dc[g.d].ranks.size() - targets.size());
    if (targets.empty()) continue;
    const Box& sb = P->src.box[size_t(g.replica)];
    const Box& db = dc[g.d].box;
    int64_t sst[RESHARD_MAX_TENSOR_NDIM], dst[RESHARD_MAX_TENSOR_NDIM];
    row_major_strides(nd, sb.shp, sst);
    row_major_strides(nd, db.shp, dst);
    int64_t s0 = 0, d0 = 0;
    for (int d = 0; d < nd; ++d) {
      s0 += (g.lo[d] - sb.off[d]) * sst[d];
      d0 += (g.lo[d] - db.off[d]) * dst[d];
    }
    if (!consumed[ri]) {
      const std::vector<int64_t> assembly = {assemble_at[g.d]};
      for (uint16_t grp : fan_groups(assemble_at[g.d] >= 0 ? assembly : targets))
        emit_box(PF, uint16_t(g.replica), grp, nd, g.ext, s0, sst, d0, dst, eb,
                 int64_t(PF.goff[grp + 1] - PF.goff[grp]));
    }
    for (int64_t r : targets)
      emit_box(PB, uint16_t(g.replica), uint16_t(r), nd, g.ext, s0, sst, d0, dst, eb);
  }
  if (too_many_groups) return fail(RESHARD_ERR_UNSUPPORTED, "more than 65535 fan-out groups");
  // replicate: each assembled destination shard, one run, to the class's other ranks
  for (size_t di = 0; di < dc.size(); ++di) {
    if (assemble_at[di] < 0) continue;
    ++S.assembled_classes;
    const int64_t vol = box_volume(nd, dc[di].box);
    const int64_t unit = 1;
    for (size_t a = 1; a < dc[di].ranks.size(); a += kMaxGroup) {
      const uint16_t grp = uint16_t(PR.goff.size() - 1);
      for (size_t b = a; b < std::min(dc[di].ranks.size(), a + size_t(kMaxGroup)); ++b)
        PR.gbuf.push_back(uint16_t(M + dc[di].ranks[b]));
      PR.goff.push_back(uint32_t(PR.gbuf.size()));
      emit_box(PR, uint16_t(M + assemble_at[di]), grp, 1, &vol, 0, &unit, 0, &unit, eb);
    }
  }
  // gather: one replica of every source class into the full tensor
  {
    std::vector<size_t> order(sc.size());
    for (size_t i = 0; i < order.size(); ++i) order[i] = i;
    std::stable_sort(order.begin(), order.end(),
                     [&](size_t a, size_t b) { return sc[a].volume > sc[b].volume; });
    std::vector<int64_t> load(size_t(M), 0);
    for (size_t ci : order) {
      int64_t best = -1;
      for (int64_t r : sc[ci].ranks)
        if (best < 0 || load[size_t(r)] < load[size_t(best)]) best = r;
      load[size_t(best)] += sc[ci].volume;
      const Box& b = sc[ci].box;
      int64_t sst[RESHARD_MAX_TENSOR_NDIM];
      row_major_strides(nd, b.shp, sst);
      int64_t d0 = 0;
      for (int d = 0; d < nd; ++d) d0 += b.off[d] * gst[d];
      emit_box(PG, uint16_t(best), 0, nd, b.shp, 0, sst, d0, gst, eb);
    }
  }
  // slice: every destination rank copies its box out of the full tensor
  for (int64_t r = 0; r < N; ++r) {
    const Box& b = P->dst.box[size_t(r)];
    if (box_volume(nd, b) == 0 || !present(P->dst_gone, r)) continue;
    int64_t dst[RESHARD_MAX_TENSOR_NDIM];
    row_major_strides(nd, b.shp, dst);
    int64_t s0 = 0;
    for (int d = 0; d < nd; ++d) s0 += b.off[d] * gst[d];
    emit_box(PS, scratch_buf, uint16_t(r), nd, b.shp, s0, gst, 0, dst, eb);
  }
  for (Program* p : {&PF, &PB, &PG, &PS, &PR}) finish_program(*p);
  PF.staged = true;
  PR.staged = true;
  for (int k = 0; k < 4; ++k) S.n_tiles[k] = int64_t(P->prog[k].tiles.size());
  S.n_replicate_tiles = int64_t(PR.tiles.size());

  // ---- traffic accounting
  for (const Program* p : {&PF, &PR})
    for (const reshard_tile_t& t : p->tiles) {
      const int64_t R = p->goff[t.dst_group + 1] - p->goff[t.dst_group];
      S.fanout_read_bytes += tile_bytes(t);
      S.fanout_write_bytes += R * tile_bytes(t);
    }
  for (const reshard_tblock_t& b : PF.tblocks) {
    PF.talign_bits |= uint64_t(b.row_bytes) | uint64_t(b.wide_off);
    for (uint32_t k = b.seg_begin; k < b.seg_begin + b.seg_count; ++k)
      PF.talign_bits |= uint64_t(PF.tsegs[k].width) | PF.tsegs[k].col |
                        uint64_t(PF.tsegs[k].narrow_off);
    const int64_t bytes = int64_t(b.row_bytes) * b.nrows;
    if (b.direction != 0) PF.tscatter = true;
    S.fanout_read_bytes += bytes;
    if (b.direction == 0) {
      S.fanout_write_bytes += bytes * int64_t(PF.goff[b.wide + 1] - PF.goff[b.wide]);
    } else {
      for (uint32_t k = b.seg_begin; k < b.seg_begin + b.seg_count; ++k) {
        const reshard_tseg_t& sg = PF.tsegs[k];
        S.fanout_write_bytes +=
            int64_t(sg.width) * b.nrows * int64_t(PF.goff[sg.narrow + 1] - PF.goff[sg.narrow]);
      }
    }
  }
  for (const reshard_tile_t& t : PB.tiles) {
    S.boxcopy_read_bytes += tile_bytes(t);
    S.boxcopy_write_bytes += tile_bytes(t);
  }
  for (const Program* p : {&PG, &PS})
    for (const reshard_tile_t& t : p->tiles) {
      S.gb_read_bytes += tile_bytes(t);
      S.gb_write_bytes += tile_bytes(t);
    }
  return RESHARD_OK;
}

}  // namespace

bool plan_live(const reshard_plan_s* plan) { return live(plan); }

reshard_status_t fail(reshard_status_t st, const std::string& msg) {
  g_last_error = msg;
  return st;
}

}  // namespace rs

using rs::fail;

namespace rs {
namespace {

// In-place declaration: source rank s is stored inside destination rank
// alias[s].  Valid when s's box lies inside that rank's box and occupies one
// contiguous range of its row-major local layout (leading dims of extent 1,
// one partial dim, trailing dims full).  Records the byte offset.
reshard_status_t read_aliases(reshard_plan_s* P, const int64_t* alias) {
  const int64_t M = P->src.nranks, N = P->dst.nranks;
  P->inplace = true;
  P->alias_dst.assign(size_t(M), -1);
  P->alias_off.assign(size_t(M), 0);
  for (int64_t s = 0; s < M; ++s) {
    const int64_t d = alias[s];
    if (d < 0) continue;
    if (d >= N) return fail(RESHARD_ERR_INVALID_ARG, "alias rank out of range");
    const Box& sb = P->src.box[size_t(s)];
    const Box& db = P->dst.box[size_t(d)];
    if (box_volume(P->ndim, sb) == 0) continue;  // nothing to hold
    int k0 = -1;
    for (int k = 0; k < P->ndim; ++k) {
      if (sb.off[k] < db.off[k] || sb.off[k] + sb.shp[k] > db.off[k] + db.shp[k])
        return fail(RESHARD_ERR_SHAPE, "source rank " + std::to_string(s) +
                                           " is not inside destination rank " + std::to_string(d));
      if (k0 < 0 && sb.shp[k] != 1) k0 = k;
    }
    for (int k = (k0 < 0 ? P->ndim : k0 + 1); k < P->ndim; ++k)
      if (sb.shp[k] != db.shp[k])
        return fail(RESHARD_ERR_SHAPE, "source rank " + std::to_string(s) +
                                           " is not one contiguous range of destination rank " +
                                           std::to_string(d));
    int64_t st[RESHARD_MAX_TENSOR_NDIM];
    row_major_strides(P->ndim, db.shp, st);
    int64_t off = 0;
    for (int k = 0; k < P->ndim; ++k) off += (sb.off[k] - db.off[k]) * st[k];
    P->alias_dst[size_t(s)] = d;
    P->alias_off[size_t(s)] = off * P->elem_bytes;
  }
  return RESHARD_OK;
}

reshard_status_t create_plan(const int64_t* global_shape, int32_t tensor_ndim,
                             reshard_dtype_t dtype, const reshard_mesh_t* src_mesh,
                             const reshard_placement_t* src_placements,
                             const reshard_mesh_t* dst_mesh,
                             const reshard_placement_t* dst_placements, const int64_t* alias,
                             reshard_plan_t* out_plan) {
  const auto t0 = std::chrono::steady_clock::now();
  TraceRange trace("reshard.plan");
  if (!out_plan) return fail(RESHARD_ERR_INVALID_ARG, "out_plan is NULL");
  *out_plan = nullptr;
  if (tensor_ndim < 1 || tensor_ndim > RESHARD_MAX_TENSOR_NDIM)
    return fail(RESHARD_ERR_UNSUPPORTED, "tensor ndim must be 1..4");
  if (!global_shape) return fail(RESHARD_ERR_INVALID_ARG, "global_shape is NULL");
  const int eb = elem_size(dtype);
  if (!eb) return fail(RESHARD_ERR_INVALID_ARG, "unknown dtype");
  int64_t numel = 1;
  for (int d = 0; d < tensor_ndim; ++d) {
    if (global_shape[d] < 0) return fail(RESHARD_ERR_INVALID_ARG, "negative global extent");
    if (global_shape[d] > 0 && numel > (int64_t(1) << 56) / global_shape[d])
      return fail(RESHARD_ERR_UNSUPPORTED, "tensor too large");
    numel *= global_shape[d];
  }
  reshard_plan_s* P = new (std::nothrow) reshard_plan_s();
  if (!P) return fail(RESHARD_ERR_NO_MEMORY, "host allocation failed");
  P->ndim = tensor_ndim;
  P->elem_bytes = eb;
  for (int d = 0; d < tensor_ndim; ++d) P->gshape[d] = global_shape[d];
  reshard_status_t st = read_layout("source", tensor_ndim, src_mesh, src_placements, &P->src);
  if (st == RESHARD_OK)
    st = read_layout("destination", tensor_ndim, dst_mesh, dst_placements, &P->dst);
  if (st == RESHARD_OK && P->src.nranks + P->dst.nranks + 1 > 65535)
    st = fail(RESHARD_ERR_UNSUPPORTED, "M + N + 1 must fit in 16 bits");
  if (st == RESHARD_OK) {
    try {
      P->src.box.resize(size_t(P->src.nranks));
      P->dst.box.resize(size_t(P->dst.nranks));
      for (int64_t r = 0; r < P->src.nranks; ++r)
        resolve_rank(P->ndim, P->gshape, P->src, r, &P->src.box[size_t(r)]);
      for (int64_t r = 0; r < P->dst.nranks; ++r)
        resolve_rank(P->ndim, P->gshape, P->dst, r, &P->dst.box[size_t(r)]);
      if (alias) st = read_aliases(P, alias);
      if (st == RESHARD_OK) st = build_plan(P);
    } catch (const std::bad_alloc&) {
      st = fail(RESHARD_ERR_NO_MEMORY, "host allocation failed while planning");
    }
  }
  if (st != RESHARD_OK) {
    delete P;
    return st;
  }
  P->magic = kPlanMagic;
  P->stats.planner_ns = std::chrono::duration_cast<std::chrono::nanoseconds>(
                            std::chrono::steady_clock::now() - t0).count();
  {
    std::lock_guard<std::mutex> lk(g_registry_mu);
    registry().insert(P);
  }
  *out_plan = P;
  return RESHARD_OK;
}

// A plan with base's layouts (and in-place declaration) and exactly the given
// ranks gone.
reshard_status_t derive_plan(const reshard_plan_s* base, const int64_t* src_gone,
                             int32_t n_src_gone, const int64_t* dst_gone, int32_t n_dst_gone,
                             reshard_plan_t* out_plan) {
  const auto t0 = std::chrono::steady_clock::now();
  TraceRange trace("reshard.plan_exclude");
  if (!out_plan) return fail(RESHARD_ERR_INVALID_ARG, "out_plan is NULL");
  *out_plan = nullptr;
  if (n_src_gone < 0 || n_dst_gone < 0 || (n_src_gone > 0 && !src_gone) ||
      (n_dst_gone > 0 && !dst_gone))
    return fail(RESHARD_ERR_INVALID_ARG, "bad rank list");
  const int64_t M = base->src.nranks, N = base->dst.nranks;
  reshard_plan_s* P = new (std::nothrow) reshard_plan_s();
  if (!P) return fail(RESHARD_ERR_NO_MEMORY, "host allocation failed");
  reshard_status_t st = RESHARD_OK;
  try {
    P->ndim = base->ndim;
    P->elem_bytes = base->elem_bytes;
    for (int d = 0; d < base->ndim; ++d) P->gshape[d] = base->gshape[d];
    P->src = base->src;
    P->dst = base->dst;
    P->inplace = base->inplace;
    P->alias_dst = base->alias_dst;
    P->alias_off = base->alias_off;
    if (n_src_gone > 0) P->src_gone.assign(size_t(M), 0);
    if (n_dst_gone > 0) P->dst_gone.assign(size_t(N), 0);
    for (int32_t i = 0; i < n_src_gone && st == RESHARD_OK; ++i) {
      if (src_gone[i] < 0 || src_gone[i] >= M) st = fail(RESHARD_ERR_INVALID_ARG, "source rank out of range");
      else P->src_gone[size_t(src_gone[i])] = 1;
    }
    for (int32_t i = 0; i < n_dst_gone && st == RESHARD_OK; ++i) {
      if (dst_gone[i] < 0 || dst_gone[i] >= N) st = fail(RESHARD_ERR_INVALID_ARG, "destination rank out of range");
      else P->dst_gone[size_t(dst_gone[i])] = 1;
    }
    // an in-place source whose own rank or host rank is gone is simply not in place
    if (st == RESHARD_OK && P->inplace)
      for (int64_t s = 0; s < M; ++s) {
        const int64_t d = P->alias_dst[size_t(s)];
        if (d >= 0 && ((!P->src_gone.empty() && P->src_gone[size_t(s)]) ||
                       (!P->dst_gone.empty() && P->dst_gone[size_t(d)])))
          P->alias_dst[size_t(s)] = -1;
      }
    if (st == RESHARD_OK) st = build_plan(P);
  } catch (const std::bad_alloc&) {
    st = fail(RESHARD_ERR_NO_MEMORY, "host allocation failed while planning");
  }
  if (st != RESHARD_OK) {
    delete P;
    return st;
  }
  P->magic = kPlanMagic;
  P->stats.planner_ns = std::chrono::duration_cast<std::chrono::nanoseconds>(
                            std::chrono::steady_clock::now() - t0).count();
  {
    std::lock_guard<std::mutex> lk(g_registry_mu);
    registry().insert(P);
  }
  *out_plan = P;
  return RESHARD_OK;
}

}  // namespace
}  // namespace rs

extern "C" {

reshard_status_t reshard_plan_exclude(reshard_plan_t plan, const int64_t* src_gone,
                                      int32_t n_src_gone, const int64_t* dst_gone,
                                      int32_t n_dst_gone, reshard_plan_t* out_plan) {
  if (out_plan) *out_plan = nullptr;
  if (!rs::live(plan)) return fail(RESHARD_ERR_BAD_HANDLE, "invalid plan handle");
  return rs::derive_plan(plan, src_gone, n_src_gone, dst_gone, n_dst_gone, out_plan);
}

reshard_status_t reshard_plan_create(const int64_t* global_shape, int32_t tensor_ndim,
                                     reshard_dtype_t dtype, const reshard_mesh_t* src_mesh,
                                     const reshard_placement_t* src_placements,
                                     const reshard_mesh_t* dst_mesh,
                                     const reshard_placement_t* dst_placements,
                                     reshard_plan_t* out_plan) {
  return rs::create_plan(global_shape, tensor_ndim, dtype, src_mesh, src_placements, dst_mesh,
                         dst_placements, nullptr, out_plan);
}

reshard_status_t reshard_plan_create_inplace(const int64_t* global_shape, int32_t tensor_ndim,
                                             reshard_dtype_t dtype, const reshard_mesh_t* src_mesh,
                                             const reshard_placement_t* src_placements,
                                             const reshard_mesh_t* dst_mesh,
                                             const reshard_placement_t* dst_placements,
                                             const int64_t* src_alias, reshard_plan_t* out_plan) {
  if (!src_alias) return fail(RESHARD_ERR_INVALID_ARG, "src_alias is NULL");
  return rs::create_plan(global_shape, tensor_ndim, dtype, src_mesh, src_placements, dst_mesh,
                         dst_placements, src_alias, out_plan);
}

reshard_status_t reshard_plan_alias(reshard_plan_t plan, int64_t src_rank, int64_t* dst_rank,
                                    int64_t* byte_offset) {
  if (!rs::live(plan)) return fail(RESHARD_ERR_BAD_HANDLE, "invalid plan handle");
  if (src_rank < 0 || src_rank >= plan->src.nranks)
    return fail(RESHARD_ERR_INVALID_ARG, "rank out of range");
  if (!dst_rank || !byte_offset) return fail(RESHARD_ERR_INVALID_ARG, "null output");
  *dst_rank = plan->inplace ? plan->alias_dst[size_t(src_rank)] : -1;
  *byte_offset = plan->inplace ? plan->alias_off[size_t(src_rank)] : 0;
  return RESHARD_OK;
}

reshard_status_t reshard_plan_destroy(reshard_plan_t plan) {
  {
    std::lock_guard<std::mutex> lk(rs::g_registry_mu);
    if (!plan || !rs::registry().erase(plan))
      return fail(RESHARD_ERR_BAD_HANDLE, "plan is NULL or already destroyed");
  }
  if (plan->d_mem) {
    int cur = -1;
    cudaGetDevice(&cur);
    if (cur != plan->device) cudaSetDevice(plan->device);
    cudaFree(plan->d_mem);
    if (cur >= 0 && cur != plan->device) cudaSetDevice(cur);
  }
  plan->magic = 0;
  delete plan;
  return RESHARD_OK;
}

reshard_status_t reshard_plan_upload(reshard_plan_t plan) {
  if (!rs::live(plan)) return fail(RESHARD_ERR_BAD_HANDLE, "invalid plan handle");
  return rs::upload_plan(plan);
}

}  // extern "C"

namespace rs {

reshard_status_t upload_plan(reshard_plan_s* plan) {
  std::lock_guard<std::mutex> lock(plan->upload_mu);
  int dev = -1;
  cudaError_t ce = cudaGetDevice(&dev);
  if (ce != cudaSuccess) return fail(RESHARD_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(ce));
  if (plan->device >= 0) {
    if (plan->device != dev)
      return fail(RESHARD_ERR_INVALID_ARG, "plan is bound to another device");
    return RESHARD_OK;
  }
  int sms = 0;
  ce = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (ce != cudaSuccess) return fail(RESHARD_ERR_CUDA, std::string("device query: ") + cudaGetErrorString(ce));
  int bps = 0;
  reshard_status_t st = rs::copy_kernel_occupancy(&bps);
  if (st != RESHARD_OK) return st;

  // one allocation: per program tiles | prefix | goff | gbuf, each 256-byte aligned
  auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
  size_t total = 0;
  size_t offs[rs::kNumPrograms][6];
  for (int k = 0; k < rs::kNumPrograms; ++k) {
    const rs::Program& p = plan->prog[k];
    const size_t sz[6] = {p.tiles.size() * sizeof(reshard_tile_t), p.prefix.size() * sizeof(int64_t),
                          p.goff.size() * sizeof(uint32_t), p.gbuf.size() * sizeof(uint16_t),
                          p.tblocks.size() * sizeof(reshard_tblock_t),
                          p.tsegs.size() * sizeof(reshard_tseg_t)};
    for (int j = 0; j < 6; ++j) {
      offs[k][j] = total;
      total += up(sz[j]);
    }
  }
  std::vector<unsigned char> host;
  try {
    host.assign(total, 0);
  } catch (const std::bad_alloc&) {
    return fail(RESHARD_ERR_NO_MEMORY, "host staging allocation failed");
  }
  for (int k = 0; k < rs::kNumPrograms; ++k) {
    const rs::Program& p = plan->prog[k];
    if (!p.tiles.empty()) std::memcpy(&host[offs[k][0]], p.tiles.data(), p.tiles.size() * sizeof(reshard_tile_t));
    if (!p.prefix.empty()) std::memcpy(&host[offs[k][1]], p.prefix.data(), p.prefix.size() * sizeof(int64_t));
    if (!p.goff.empty()) std::memcpy(&host[offs[k][2]], p.goff.data(), p.goff.size() * sizeof(uint32_t));
    if (!p.gbuf.empty()) std::memcpy(&host[offs[k][3]], p.gbuf.data(), p.gbuf.size() * sizeof(uint16_t));
    if (!p.tblocks.empty())
      std::memcpy(&host[offs[k][4]], p.tblocks.data(), p.tblocks.size() * sizeof(reshard_tblock_t));
    if (!p.tsegs.empty())
      std::memcpy(&host[offs[k][5]], p.tsegs.data(), p.tsegs.size() * sizeof(reshard_tseg_t));
  }
  void* d = nullptr;
  ce = cudaMalloc(&d, std::max<size_t>(total, 256));
  if (ce != cudaSuccess) return fail(RESHARD_ERR_NO_MEMORY, std::string("cudaMalloc: ") + cudaGetErrorString(ce));
  ce = cudaMemcpy(d, host.data(), total, cudaMemcpyHostToDevice);
  if (ce != cudaSuccess) {
    cudaFree(d);
    return fail(RESHARD_ERR_CUDA, std::string("cudaMemcpy: ") + cudaGetErrorString(ce));
  }
  unsigned char* base = static_cast<unsigned char*>(d);
  for (int k = 0; k < rs::kNumPrograms; ++k) {
    rs::Program& p = plan->prog[k];
    p.d_tiles = reinterpret_cast<const reshard_tile_t*>(base + offs[k][0]);
    p.d_prefix = reinterpret_cast<const int64_t*>(base + offs[k][1]);
    p.d_goff = reinterpret_cast<const uint32_t*>(base + offs[k][2]);
    p.d_gbuf = reinterpret_cast<const uint16_t*>(base + offs[k][3]);
    p.d_tblocks = reinterpret_cast<const reshard_tblock_t*>(base + offs[k][4]);
    p.d_tsegs = reinterpret_cast<const reshard_tseg_t*>(base + offs[k][5]);
  }
  plan->d_mem = d;
  plan->device = dev;
  plan->num_sms = sms;
  plan->blocks_per_sm = bps;
  return RESHARD_OK;
}

}  // namespace rs


namespace rs {

// Build the buffer table [src..., dst..., scratch] into out[M + N + 1] and check
// null pointers (a NULL pointer is accepted for an empty shard and for a rank an
// excluded plan leaves out) and, for in-place plans, the source aliases.
reshard_status_t buffer_table(reshard_plan_t plan, const void* const* src_ptrs,
                              void* const* dst_ptrs, void* scratch, unsigned char** out,
                              int64_t capacity) {
  const int64_t M = plan->src.nranks, N = plan->dst.nranks;
  if (M + N + 1 > RESHARD_MAX_EXEC_BUFFERS || M + N + 1 > capacity)
    return fail(RESHARD_ERR_UNSUPPORTED, "M + N + 1 exceeds RESHARD_MAX_EXEC_BUFFERS");
  if (!src_ptrs || !dst_ptrs) return fail(RESHARD_ERR_INVALID_ARG, "null pointer array");
  unsigned char** const b = out;
  for (int64_t r = 0; r < M; ++r) {
    if (!src_ptrs[r] && rs::box_volume(plan->ndim, plan->src.box[size_t(r)]) > 0 &&
        (plan->src_gone.empty() || !plan->src_gone[size_t(r)]))
      return fail(RESHARD_ERR_INVALID_ARG, "NULL source pointer for a non-empty shard (rank " +
                                               std::to_string(r) + ")");
    b[r] = static_cast<unsigned char*>(const_cast<void*>(src_ptrs[r]));
  }
  for (int64_t r = 0; r < N; ++r) {
    if (!dst_ptrs[r] && rs::box_volume(plan->ndim, plan->dst.box[size_t(r)]) > 0 &&
        (plan->dst_gone.empty() || !plan->dst_gone[size_t(r)]))
      return fail(RESHARD_ERR_INVALID_ARG, "NULL destination pointer for a non-empty shard (rank " +
                                               std::to_string(r) + ")");
    b[M + r] = static_cast<unsigned char*>(dst_ptrs[r]);
  }
  b[M + N] = static_cast<unsigned char*>(scratch);
  if (plan->inplace) {
    for (int64_t r = 0; r < M; ++r) {
      const int64_t d = plan->alias_dst[size_t(r)];
      if (d < 0) continue;
      if (b[r] != b[M + d] + plan->alias_off[size_t(r)])
        return fail(RESHARD_ERR_INVALID_ARG,
                    "in-place plan: source rank " + std::to_string(r) +
                        " must point into destination rank " + std::to_string(d) +
                        " at byte offset " + std::to_string(plan->alias_off[size_t(r)]));
    }
  }
  return RESHARD_OK;
}

reshard_status_t buffer_table(reshard_plan_t plan, const void* const* src_ptrs,
                              void* const* dst_ptrs, void* scratch, std::vector<unsigned char*>* bufs) {
  const int64_t n = plan->src.nranks + plan->dst.nranks + 1;
  if (n > RESHARD_MAX_EXEC_BUFFERS)
    return fail(RESHARD_ERR_UNSUPPORTED, "M + N + 1 exceeds RESHARD_MAX_EXEC_BUFFERS");
  bufs->resize(size_t(n));
  return buffer_table(plan, src_ptrs, dst_ptrs, scratch, bufs->data(), n);
}

}  // namespace rs

extern "C" {

reshard_status_t reshard_execute_ex(reshard_plan_t plan, const void* const* src_ptrs,
                                    void* const* dst_ptrs, int32_t kernel, void* stream) {
  rs::TraceRange trace("reshard.exec");
  if (!rs::live(plan)) return fail(RESHARD_ERR_BAD_HANDLE, "invalid plan handle");
  if (kernel != RESHARD_KERNEL_FANOUT && kernel != RESHARD_KERNEL_BOXCOPY)
    return fail(RESHARD_ERR_INVALID_ARG, "unknown kernel");
  std::vector<unsigned char*> bufs;
  reshard_status_t st = rs::buffer_table(plan, src_ptrs, dst_ptrs, nullptr, &bufs);
  if (st != RESHARD_OK) return st;
  st = reshard_plan_upload(plan);
  if (st != RESHARD_OK) return st;
  if (kernel == RESHARD_KERNEL_FANOUT) return rs::launch_fanout(plan, bufs.data(), int(bufs.size()), stream);
  return rs::launch_program(plan, plan->prog[RESHARD_PROGRAM_BOXCOPY], bufs.data(), int(bufs.size()),
                            stream);
}

reshard_status_t reshard_plan_path(reshard_plan_t plan, const void* const* src_ptrs,
                                   void* const* dst_ptrs, int32_t kernel, int32_t* path,
                                   int32_t* width) {
  if (!rs::live(plan)) return fail(RESHARD_ERR_BAD_HANDLE, "invalid plan handle");
  if (kernel != RESHARD_KERNEL_FANOUT && kernel != RESHARD_KERNEL_BOXCOPY)
    return fail(RESHARD_ERR_INVALID_ARG, "unknown kernel");
  std::vector<unsigned char*> bufs;
  reshard_status_t st = rs::buffer_table(plan, src_ptrs, dst_ptrs, nullptr, &bufs);
  if (st != RESHARD_OK) return st;
  if (bufs.size() > size_t(RESHARD_MAX_EXEC_BUFFERS))
    return fail(RESHARD_ERR_UNSUPPORTED, "too many buffers");
  const rs::Program& p =
      plan->prog[kernel == RESHARD_KERNEL_FANOUT ? RESHARD_PROGRAM_FANOUT : RESHARD_PROGRAM_BOXCOPY];
  const rs::Dispatch d = rs::decide(p, bufs.data(), int(bufs.size()), true);
  if (path) *path = d.path;
  if (width) *width = 1 << d.w_log2;
  return RESHARD_OK;
}

reshard_status_t reshard_execute(reshard_plan_t plan, const void* const* src_ptrs,
                                 void* const* dst_ptrs, void* stream) {
  return reshard_execute_ex(plan, src_ptrs, dst_ptrs, RESHARD_KERNEL_FANOUT, stream);
}

reshard_status_t gather_broadcast_execute(reshard_plan_t plan, const void* const* src_ptrs,
                                          void* const* dst_ptrs, void* full_scratch,
                                          size_t scratch_bytes, void* stream) {
  rs::TraceRange trace("gb.exec");
  if (!rs::live(plan)) return fail(RESHARD_ERR_BAD_HANDLE, "invalid plan handle");
  if (plan->stats.global_bytes > 0) {
    if (!full_scratch) return fail(RESHARD_ERR_INVALID_ARG, "full_scratch is NULL");
    if (scratch_bytes < size_t(plan->stats.global_bytes))
      return fail(RESHARD_ERR_INVALID_ARG, "full_scratch is smaller than the global tensor");
  }
  std::vector<unsigned char*> bufs;
  reshard_status_t st = rs::buffer_table(plan, src_ptrs, dst_ptrs, full_scratch, &bufs);
  if (st != RESHARD_OK) return st;
  st = reshard_plan_upload(plan);
  if (st != RESHARD_OK) return st;
  st = rs::launch_program(plan, plan->prog[RESHARD_PROGRAM_GATHER], bufs.data(), int(bufs.size()), stream);
  if (st != RESHARD_OK) return st;
  return rs::launch_program(plan, plan->prog[RESHARD_PROGRAM_SLICE], bufs.data(), int(bufs.size()), stream);
}

reshard_status_t reshard_plan_local_shape(reshard_plan_t plan, int32_t side, int64_t rank,
                                          int64_t* shape, int64_t* offset) {
  if (!rs::live(plan)) return fail(RESHARD_ERR_BAD_HANDLE, "invalid plan handle");
  if (side != 0 && side != 1) return fail(RESHARD_ERR_INVALID_ARG, "side must be 0 or 1");
  const rs::Layout& L = side == 0 ? plan->src : plan->dst;
  if (rank < 0 || rank >= L.nranks) return fail(RESHARD_ERR_INVALID_ARG, "rank out of range");
  if (!shape && !offset) return fail(RESHARD_ERR_INVALID_ARG, "both outputs are NULL");
  for (int d = 0; d < plan->ndim; ++d) {
    if (shape) shape[d] = L.box[size_t(rank)].shp[d];
    if (offset) offset[d] = L.box[size_t(rank)].off[d];
  }
  return RESHARD_OK;
}

reshard_status_t reshard_plan_stats(reshard_plan_t plan, reshard_stats_t* out) {
  if (!rs::live(plan)) return fail(RESHARD_ERR_BAD_HANDLE, "invalid plan handle");
  if (!out) return fail(RESHARD_ERR_INVALID_ARG, "out is NULL");
  *out = plan->stats;
  return RESHARD_OK;
}

reshard_status_t reshard_plan_program(reshard_plan_t plan, int32_t program,
                                      const reshard_tile_t** tiles, int64_t* ntiles,
                                      const int64_t** unit_prefix, const uint32_t** group_offsets,
                                      const uint16_t** group_buffers, int64_t* ngroups) {
  if (!rs::live(plan)) return fail(RESHARD_ERR_BAD_HANDLE, "invalid plan handle");
  if (program < 0 || program >= rs::kNumPrograms)
    return fail(RESHARD_ERR_INVALID_ARG, "unknown program");
  const rs::Program& p = plan->prog[program];
  if (tiles) *tiles = p.tiles.data();
  if (ntiles) *ntiles = int64_t(p.tiles.size());
  if (unit_prefix) *unit_prefix = p.prefix.data();
  if (group_offsets) *group_offsets = p.goff.data();
  if (group_buffers) *group_buffers = p.gbuf.data();
  if (ngroups) *ngroups = int64_t(p.goff.size()) - 1;
  return RESHARD_OK;
}

reshard_status_t reshard_plan_transposes(reshard_plan_t plan, int32_t program,
                                         const reshard_tblock_t** blocks, int64_t* nblocks,
                                         const reshard_tseg_t** segs, int64_t* nsegs) {
  if (!rs::live(plan)) return fail(RESHARD_ERR_BAD_HANDLE, "invalid plan handle");
  if (program < 0 || program >= rs::kNumPrograms)
    return fail(RESHARD_ERR_INVALID_ARG, "unknown program");
  const rs::Program& p = plan->prog[program];
  if (blocks) *blocks = p.tblocks.data();
  if (nblocks) *nblocks = int64_t(p.tblocks.size());
  if (segs) *segs = p.tsegs.data();
  if (nsegs) *nsegs = int64_t(p.tsegs.size());
  return RESHARD_OK;
}

int64_t reshard_tile_units(const reshard_tile_t* tile) {
  return tile ? rs::tile_units(*tile) : 0;
}

const char* reshard_last_error(void) { return rs::g_last_error.c_str(); }

const char* reshard_version(void) { return "libreshard 0.1 (sm_103a)"; }

}  // extern "C"
