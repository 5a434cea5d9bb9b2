// batch.cpp -- few launches for the fan-out programs of many plans (a whole
// model's refit).  The plans that take the TMA fan-out with 16-byte-aligned
// buffers (and have no transpose blocks) form one class: their tiles are
// concatenated into one program over a combined buffer table [plan 0 sources,
// plan 0 destinations, plan 1 ...], and the fan-out kernel's work queue
// spreads the whole class evenly over the GPU, with no launch boundary (and no
// ramp-down tail) between tensors.  Every other plan is a class of its own and
// runs as reshard_execute runs it: the other kernels split their work into
// equal static ranges, and tensors whose rows cost different amounts per byte
// (2-byte rows against kilobyte rows) were measured up to 36x slower
// concatenated than launched one by one.  A merged class whose buffers turn
// out less aligned than assumed runs its plans one by one too.
#include <cuda_runtime.h>

#include <algorithm>
#include <memory>
#include <mutex>
#include <new>
#include <string>
#include <unordered_set>
#include <vector>

#include "internal.h"

namespace rs {
namespace {

// A class: one plan on its own (solo), or TMA fan-out plans concatenated.
struct BatchClass {
  bool solo = true;
  std::vector<int32_t> members;  // plan indices, in batch order
  std::vector<int64_t> base;     // first buffer index of each member in the class table
  int64_t nbufs = 0;
  reshard_plan_s combined;       // merged: prog[RESHARD_PROGRAM_FANOUT] is the concatenation
};

// Does the plan take the TMA fan-out with 16-byte-aligned buffers?
bool mergeable(const Program& F) {
  if (!F.tblocks.empty()) return false;
  std::vector<unsigned char*> zeros(RESHARD_MAX_EXEC_BUFFERS, nullptr);  // aligned, congruent
  return decide(F, zeros.data(), int(zeros.size()), true).path == RESHARD_PATH_TMA_FANOUT;
}

// Appends a plan's fan-out program (its buffers from `base` on) to C.
void append_plan(Program& C, const Program& F, int64_t base) {
  const int64_t gbase = int64_t(C.goff.size()) - 1;
  for (size_t g = 0; g + 1 < F.goff.size(); ++g) {
    for (uint32_t k = F.goff[g]; k < F.goff[g + 1]; ++k)
      C.gbuf.push_back(uint16_t(base + F.gbuf[k]));
    C.goff.push_back(uint32_t(C.gbuf.size()));
  }
  for (reshard_tile_t t : F.tiles) {
    t.src_buf = uint16_t(base + t.src_buf);
    t.dst_group = uint16_t(gbase + t.dst_group);
    C.tiles.push_back(t);
  }
  const uint32_t sbase = uint32_t(C.tsegs.size());
  for (reshard_tblock_t b : F.tblocks) {
    b.wide = uint16_t(b.direction == 0 ? gbase + b.wide : base + b.wide);
    b.seg_begin += sbase;
    C.tblocks.push_back(b);
  }
  for (const reshard_tblock_t& b : F.tblocks) {
    for (uint32_t j = b.seg_begin; j < b.seg_begin + b.seg_count; ++j) {
      reshard_tseg_t sg = F.tsegs[j];
      sg.narrow = uint16_t(b.direction == 0 ? base + sg.narrow : gbase + sg.narrow);
      C.tsegs.push_back(sg);
    }
  }
  C.align_bits |= F.align_bits;
  C.has_planes = C.has_planes || F.has_planes;
  C.max_fanout = std::max(C.max_fanout, F.max_fanout);
  C.tile_bytes += F.tile_bytes;
  C.write_bytes += F.write_bytes;
  C.talign_bits |= F.talign_bits;
  C.tscatter = C.tscatter || F.tscatter;
  C.long_row_bytes += F.long_row_bytes;
  C.wide_row_bytes += F.wide_row_bytes;
  C.narrow_row_bytes += F.narrow_row_bytes;
}

void finish_class(BatchClass& c) {
  Program& C = c.combined.prog[RESHARD_PROGRAM_FANOUT];
  C.prefix.assign(C.tiles.size() + 1, 0);
  for (size_t i = 0; i < C.tiles.size(); ++i) C.prefix[i + 1] = C.prefix[i] + tile_units(C.tiles[i]);
  C.staged = true;
}

std::mutex g_batch_mu;

}  // namespace
}  // namespace rs

struct reshard_batch_s {
  std::vector<reshard_plan_t> plans;
  std::vector<std::unique_ptr<rs::BatchClass>> classes;
};

namespace rs {
namespace {

std::unordered_set<const reshard_batch_s*>& batches() {
  static std::unordered_set<const reshard_batch_s*> b;
  return b;
}
bool batch_live(const reshard_batch_s* b) {
  if (!b) return false;
  std::lock_guard<std::mutex> lk(g_batch_mu);
  return batches().count(b) != 0;
}

void free_batch(reshard_batch_s* B) {
  for (auto& c : B->classes) {
    reshard_plan_s& P = c->combined;
    if (!P.d_mem) continue;
    int cur = -1;
    cudaGetDevice(&cur);
    if (cur != P.device) cudaSetDevice(P.device);
    cudaFree(P.d_mem);
    P.d_mem = nullptr;
    if (cur >= 0 && cur != P.device) cudaSetDevice(cur);
  }
  delete B;
}

}  // namespace
}  // namespace rs

using rs::fail;

extern "C" {

reshard_status_t reshard_batch_create(const reshard_plan_t* plans, int32_t nplans,
                                      reshard_batch_t* out_batch) {
  if (!out_batch) return fail(RESHARD_ERR_INVALID_ARG, "out_batch is NULL");
  *out_batch = nullptr;
  if (!plans || nplans < 1) return fail(RESHARD_ERR_INVALID_ARG, "no plans");
  reshard_batch_s* B = new (std::nothrow) reshard_batch_s();
  if (!B) return fail(RESHARD_ERR_NO_MEMORY, "host allocation failed");
  try {
    rs::BatchClass* open = nullptr;  // the merged class still taking plans
    for (int32_t i = 0; i < nplans; ++i) {
      reshard_plan_s* p = plans[i];
      if (!rs::plan_live(p)) {
        rs::free_batch(B);
        return fail(RESHARD_ERR_BAD_HANDLE, "plan " + std::to_string(i) + " is not a live plan");
      }
      B->plans.push_back(p);
      const rs::Program& F = p->prog[RESHARD_PROGRAM_FANOUT];
      if (F.total_units() == 0 && F.tblocks.empty()) continue;  // nothing to copy
      const int64_t nb = p->src.nranks + p->dst.nranks;
      if (nb + 1 > RESHARD_MAX_EXEC_BUFFERS) {
        rs::free_batch(B);
        return fail(RESHARD_ERR_UNSUPPORTED, "plan " + std::to_string(i) +
                                                 " has more ranks than one launch can address");
      }
      if (!rs::mergeable(F) || !p->prog[RESHARD_PROGRAM_REPLICATE].tiles.empty()) {
        B->classes.emplace_back(new rs::BatchClass());
        B->classes.back()->members.push_back(i);
        continue;
      }
      // a launch addresses at most RESHARD_MAX_EXEC_BUFFERS buffers and 65535 groups
      if (open && (open->nbufs + nb + 1 > RESHARD_MAX_EXEC_BUFFERS ||
                   open->combined.prog[RESHARD_PROGRAM_FANOUT].goff.size() + F.goff.size() > 65537))
        open = nullptr;
      if (!open) {
        B->classes.emplace_back(new rs::BatchClass());
        open = B->classes.back().get();
        open->solo = false;
        open->combined.prog[RESHARD_PROGRAM_FANOUT].goff.push_back(0);
      }
      open->members.push_back(i);
      open->base.push_back(open->nbufs);
      rs::append_plan(open->combined.prog[RESHARD_PROGRAM_FANOUT], F, open->nbufs);
      open->nbufs += nb;
    }
    for (auto& c : B->classes)
      if (!c->solo) rs::finish_class(*c);
  } catch (const std::bad_alloc&) {
    rs::free_batch(B);
    return fail(RESHARD_ERR_NO_MEMORY, "host allocation failed while batching");
  }
  {
    std::lock_guard<std::mutex> lk(rs::g_batch_mu);
    rs::batches().insert(B);
  }
  *out_batch = B;
  return RESHARD_OK;
}

reshard_status_t reshard_batch_classes(reshard_batch_t batch, int32_t* nclasses,
                                       int32_t* plan_class) {
  if (!rs::batch_live(batch)) return fail(RESHARD_ERR_BAD_HANDLE, "invalid batch handle");
  if (nclasses) *nclasses = int32_t(batch->classes.size());
  if (plan_class) {
    std::fill(plan_class, plan_class + batch->plans.size(), -1);
    for (size_t k = 0; k < batch->classes.size(); ++k)
      for (int32_t i : batch->classes[k]->members) plan_class[i] = int32_t(k);
  }
  return RESHARD_OK;
}

reshard_status_t reshard_batch_execute(reshard_batch_t batch, const void* const* const* src_ptrs,
                                       void* const* const* dst_ptrs, void* stream) {
  rs::TraceRange trace("reshard.batch_exec");
  if (!rs::batch_live(batch)) return fail(RESHARD_ERR_BAD_HANDLE, "invalid batch handle");
  if (!src_ptrs || !dst_ptrs) return fail(RESHARD_ERR_INVALID_ARG, "null pointer array");
  const size_t n = batch->plans.size();
  // every plan's buffer table (and argument checks) before anything is launched
  std::vector<std::vector<unsigned char*>> tables(n);
  for (size_t i = 0; i < n; ++i) {
    reshard_plan_s* p = batch->plans[i];
    if (!rs::plan_live(p))
      return fail(RESHARD_ERR_BAD_HANDLE, "plan " + std::to_string(i) + " was destroyed");
    reshard_status_t st = rs::buffer_table(p, src_ptrs[i], dst_ptrs[i], nullptr, &tables[i]);
    if (st != RESHARD_OK) return st;
  }
  for (auto& cp : batch->classes) {
    rs::BatchClass& c = *cp;
    if (c.solo) {
      // as reshard_execute, with the buffer table built above
      reshard_plan_s* p = batch->plans[size_t(c.members[0])];
      const std::vector<unsigned char*>& t = tables[size_t(c.members[0])];
      reshard_status_t st = reshard_plan_upload(p);
      if (st != RESHARD_OK) return st;
      st = rs::launch_fanout(p, t.data(), int(t.size()), stream);
      if (st != RESHARD_OK) return st;
      continue;
    }
    std::vector<unsigned char*> flat(size_t(c.nbufs) + 1, nullptr);
    for (size_t k = 0; k < c.members.size(); ++k) {
      const std::vector<unsigned char*>& t = tables[size_t(c.members[k])];
      std::copy(t.begin(), t.end() - 1, flat.begin() + c.base[k]);  // without the scratch slot
    }
    const rs::Program& C = c.combined.prog[RESHARD_PROGRAM_FANOUT];
    uint64_t align = C.align_bits;
    for (unsigned char* b : flat) align |= reinterpret_cast<uint64_t>(b);
    if ((align & 15u) != 0) {
      // the buffers are not all 16-byte aligned: each plan picks its own kernel
      for (int32_t i : c.members) {
        reshard_status_t st = reshard_execute(batch->plans[size_t(i)], src_ptrs[i], dst_ptrs[i], stream);
        if (st != RESHARD_OK) return st;
      }
      continue;
    }
    reshard_status_t st = rs::upload_plan(&c.combined);
    if (st != RESHARD_OK) return st;
    st = rs::launch_program(&c.combined, C, flat.data(), int(flat.size()), stream);
    if (st != RESHARD_OK) return st;
  }
  return RESHARD_OK;
}

reshard_status_t reshard_batch_destroy(reshard_batch_t batch) {
  {
    std::lock_guard<std::mutex> lk(rs::g_batch_mu);
    if (!batch || !rs::batches().erase(batch))
      return fail(RESHARD_ERR_BAD_HANDLE, "batch is NULL or already destroyed");
  }
  rs::free_batch(batch);
  return RESHARD_OK;
}

}  // extern "C"
