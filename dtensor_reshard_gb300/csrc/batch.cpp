// batch.cpp -- one launch for the fan-out programs of many plans (a whole
// model's refit).  The plans' tiles are concatenated into one program over a
// combined buffer table [plan 0 sources, plan 0 destinations, plan 1 ...];
// the work-unit partition then spreads the whole model evenly over the GPU,
// with no launch boundary (and no ramp-down tail) between tensors.
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>
#include <new>
#include <string>
#include <unordered_set>
#include <vector>

#include "internal.h"

struct reshard_batch_s {
  std::vector<reshard_plan_t> plans;
  std::vector<int64_t> base;  // first buffer index of each plan in the combined table
  int64_t nbufs = 0;
  reshard_plan_s combined;    // prog[RESHARD_PROGRAM_FANOUT] holds the concatenated program
};

namespace rs {
namespace {

std::mutex g_batch_mu;
std::unordered_set<const reshard_batch_s*>& batches() {
  static std::unordered_set<const reshard_batch_s*> b;
  return b;
}
bool batch_live(const reshard_batch_s* b) {
  if (!b) return false;
  std::lock_guard<std::mutex> lk(g_batch_mu);
  return batches().count(b) != 0;
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
  rs::Program& C = B->combined.prog[RESHARD_PROGRAM_FANOUT];
  try {
    C.goff.push_back(0);
    for (int32_t i = 0; i < nplans; ++i) {
      reshard_plan_s* p = plans[i];
      if (!rs::plan_live(p)) {
        delete B;
        return fail(RESHARD_ERR_BAD_HANDLE, "plan " + std::to_string(i) + " is not a live plan");
      }
      const int64_t base = B->nbufs;
      const int64_t nb = p->src.nranks + p->dst.nranks;
      if (base + nb + 1 > RESHARD_MAX_EXEC_BUFFERS) {
        delete B;
        return fail(RESHARD_ERR_UNSUPPORTED,
                    "the plans' ranks exceed RESHARD_MAX_EXEC_BUFFERS; split the batch");
      }
      const rs::Program& F = p->prog[RESHARD_PROGRAM_FANOUT];
      const int64_t gbase = int64_t(C.goff.size()) - 1;
      if (gbase + int64_t(F.goff.size()) > 65536) {
        delete B;
        return fail(RESHARD_ERR_UNSUPPORTED, "more than 65535 fan-out groups in the batch");
      }
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
      for (size_t k = 0; k < F.tblocks.size(); ++k) {
        const reshard_tblock_t& b = F.tblocks[k];
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
      C.long_row_bytes += F.long_row_bytes;
      C.wide_row_bytes += F.wide_row_bytes;
      B->plans.push_back(p);
      B->base.push_back(base);
      B->nbufs = base + nb;
    }
    C.prefix.assign(C.tiles.size() + 1, 0);
    for (size_t i = 0; i < C.tiles.size(); ++i)
      C.prefix[i + 1] = C.prefix[i] + rs::tile_units(C.tiles[i]);
    C.staged = true;
  } catch (const std::bad_alloc&) {
    delete B;
    return fail(RESHARD_ERR_NO_MEMORY, "host allocation failed while batching");
  }
  {
    std::lock_guard<std::mutex> lk(rs::g_batch_mu);
    rs::batches().insert(B);
  }
  *out_batch = B;
  return RESHARD_OK;
}

reshard_status_t reshard_batch_execute(reshard_batch_t batch, const void* const* const* src_ptrs,
                                       void* const* const* dst_ptrs, void* stream) {
  rs::TraceRange trace("reshard.batch_exec");
  if (!rs::batch_live(batch)) return fail(RESHARD_ERR_BAD_HANDLE, "invalid batch handle");
  if (!src_ptrs || !dst_ptrs) return fail(RESHARD_ERR_INVALID_ARG, "null pointer array");
  const size_t n = batch->plans.size();
  std::vector<unsigned char*> flat(size_t(batch->nbufs) + 1, nullptr);
  std::vector<unsigned char*> one;
  for (size_t i = 0; i < n; ++i) {
    reshard_plan_s* p = batch->plans[i];
    if (!rs::plan_live(p))
      return fail(RESHARD_ERR_BAD_HANDLE, "plan " + std::to_string(i) + " was destroyed");
    reshard_status_t st = rs::buffer_table(p, src_ptrs[i], dst_ptrs[i], nullptr, &one);
    if (st != RESHARD_OK) return st;
    std::copy(one.begin(), one.end() - 1, flat.begin() + batch->base[i]);
  }
  const rs::Program& C = batch->combined.prog[RESHARD_PROGRAM_FANOUT];
  uint64_t align = C.align_bits;
  for (unsigned char* b : flat) align |= reinterpret_cast<uint64_t>(b);
  if ((align & 15u) != 0) {
    // not every tile can take 16-byte copies: each plan picks its own kernel
    for (size_t i = 0; i < n; ++i) {
      reshard_status_t st = reshard_execute(batch->plans[i], src_ptrs[i], dst_ptrs[i], stream);
      if (st != RESHARD_OK) return st;
    }
    return RESHARD_OK;
  }
  reshard_status_t st = rs::upload_plan(&batch->combined);
  if (st != RESHARD_OK) return st;
  return rs::launch_program(&batch->combined, C, flat.data(), int(flat.size()), stream);
}

reshard_status_t reshard_batch_destroy(reshard_batch_t batch) {
  {
    std::lock_guard<std::mutex> lk(rs::g_batch_mu);
    if (!batch || !rs::batches().erase(batch))
      return fail(RESHARD_ERR_BAD_HANDLE, "batch is NULL or already destroyed");
  }
  if (batch->combined.d_mem) {
    int cur = -1;
    cudaGetDevice(&cur);
    if (cur != batch->combined.device) cudaSetDevice(batch->combined.device);
    cudaFree(batch->combined.d_mem);
    if (cur >= 0 && cur != batch->combined.device) cudaSetDevice(cur);
  }
  delete batch;
  return RESHARD_OK;
}

}  // extern "C"
