// refit.cpp -- one call for a whole model's weight refit.  Every plan is routed
// either to the read-once reshard or to gather-and-broadcast (the hybrid split
// of "Integracio es hibrid megoldas a NeMo RL-ben", news.bpdata.com: the
// feed-forward projections through the Reshard collective, small irregular
// weights through gather-and-broadcast); the reshard group can go out as one
// batch launch, and the gather-and-broadcast group shares one scratch buffer,
// used tensor after tensor in stream order.
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>
#include <new>
#include <string>
#include <unordered_set>
#include <vector>

#include "internal.h"

struct reshard_refit_s {
  std::vector<reshard_plan_t> plans;
  std::vector<int32_t> routes;        // resolved: RESHARD or GATHER_BROADCAST
  std::vector<int32_t> reshard_idx;   // plans on the reshard path, in order
  std::vector<int32_t> gb_idx;        // plans on gather-and-broadcast, in order
  uint64_t scratch_bytes = 0;         // largest global tensor among gb_idx
  reshard_batch_t batch = nullptr;    // reshard_idx as one batch (RESHARD_REFIT_BATCH)
};

namespace rs {
namespace {

std::mutex g_refit_mu;
std::unordered_set<const reshard_refit_s*>& refits() {
  static std::unordered_set<const reshard_refit_s*> r;
  return r;
}
bool refit_live(const reshard_refit_s* r) {
  if (!r) return false;
  std::lock_guard<std::mutex> lk(g_refit_mu);
  return refits().count(r) != 0;
}

}  // namespace
}  // namespace rs

using rs::fail;

extern "C" {

reshard_status_t reshard_refit_create(const reshard_plan_t* plans, const int32_t* routes,
                                      int32_t nplans, uint32_t flags, reshard_refit_t* out_refit) {
  if (!out_refit) return fail(RESHARD_ERR_INVALID_ARG, "out_refit is NULL");
  *out_refit = nullptr;
  if (!plans || nplans < 1) return fail(RESHARD_ERR_INVALID_ARG, "no plans");
  if ((flags & ~uint32_t(RESHARD_REFIT_BATCH)) != 0)
    return fail(RESHARD_ERR_INVALID_ARG, "unknown refit flags");
  reshard_refit_s* R = new (std::nothrow) reshard_refit_s();
  if (!R) return fail(RESHARD_ERR_NO_MEMORY, "host allocation failed");
  try {
    for (int32_t i = 0; i < nplans; ++i) {
      if (!rs::plan_live(plans[i])) {
        delete R;
        return fail(RESHARD_ERR_BAD_HANDLE, "plan " + std::to_string(i) + " is not a live plan");
      }
      int32_t route = routes ? routes[i] : RESHARD_ROUTE_AUTO;
      if (route < RESHARD_ROUTE_AUTO || route > RESHARD_ROUTE_GATHER_BROADCAST) {
        delete R;
        return fail(RESHARD_ERR_INVALID_ARG, "plan " + std::to_string(i) + ": unknown route");
      }
      // On one GPU the reshard reads G and writes D bytes in one launch, gather-and-
      // broadcast moves 2G + 2D in two: AUTO always takes the reshard.
      if (route == RESHARD_ROUTE_AUTO) route = RESHARD_ROUTE_RESHARD;
      R->plans.push_back(plans[i]);
      R->routes.push_back(route);
      if (route == RESHARD_ROUTE_RESHARD) {
        R->reshard_idx.push_back(i);
      } else {
        R->gb_idx.push_back(i);
        R->scratch_bytes = std::max<uint64_t>(R->scratch_bytes,
                                              uint64_t(plans[i]->stats.global_bytes));
      }
    }
    if ((flags & RESHARD_REFIT_BATCH) && !R->reshard_idx.empty()) {
      std::vector<reshard_plan_t> group;
      for (int32_t i : R->reshard_idx) group.push_back(plans[i]);
      reshard_status_t st = reshard_batch_create(group.data(), int32_t(group.size()), &R->batch);
      if (st != RESHARD_OK) {
        delete R;
        return st;
      }
    }
  } catch (const std::bad_alloc&) {
    if (R->batch) reshard_batch_destroy(R->batch);
    delete R;
    return fail(RESHARD_ERR_NO_MEMORY, "host allocation failed while routing");
  }
  {
    std::lock_guard<std::mutex> lk(rs::g_refit_mu);
    rs::refits().insert(R);
  }
  *out_refit = R;
  return RESHARD_OK;
}

reshard_status_t reshard_refit_info(reshard_refit_t refit, int32_t* routes, uint64_t* scratch_bytes) {
  if (!rs::refit_live(refit)) return fail(RESHARD_ERR_BAD_HANDLE, "invalid refit handle");
  if (routes) std::copy(refit->routes.begin(), refit->routes.end(), routes);
  if (scratch_bytes) *scratch_bytes = refit->scratch_bytes;
  return RESHARD_OK;
}

reshard_status_t reshard_refit_execute(reshard_refit_t refit, const void* const* const* src_ptrs,
                                       void* const* const* dst_ptrs, void* scratch,
                                       size_t scratch_bytes, void* stream) {
  rs::TraceRange trace("reshard.refit_exec");
  if (!rs::refit_live(refit)) return fail(RESHARD_ERR_BAD_HANDLE, "invalid refit handle");
  if (!src_ptrs || !dst_ptrs) return fail(RESHARD_ERR_INVALID_ARG, "null pointer array");
  if (!refit->gb_idx.empty() && refit->scratch_bytes > 0) {
    if (!scratch) return fail(RESHARD_ERR_INVALID_ARG, "scratch is NULL");
    if (scratch_bytes < refit->scratch_bytes)
      return fail(RESHARD_ERR_INVALID_ARG, "scratch is smaller than the largest gathered tensor");
  }
  for (size_t i = 0; i < refit->plans.size(); ++i)
    if (!rs::plan_live(refit->plans[i]))
      return fail(RESHARD_ERR_BAD_HANDLE, "plan " + std::to_string(i) + " was destroyed");
  reshard_status_t st = RESHARD_OK;
  if (refit->batch) {
    std::vector<const void* const*> s;
    std::vector<void* const*> d;
    for (int32_t i : refit->reshard_idx) {
      s.push_back(src_ptrs[i]);
      d.push_back(dst_ptrs[i]);
    }
    st = reshard_batch_execute(refit->batch, s.data(), d.data(), stream);
    if (st != RESHARD_OK) return st;
  } else {
    for (int32_t i : refit->reshard_idx) {
      st = reshard_execute(refit->plans[size_t(i)], src_ptrs[i], dst_ptrs[i], stream);
      if (st != RESHARD_OK) return st;
    }
  }
  for (int32_t i : refit->gb_idx) {
    st = gather_broadcast_execute(refit->plans[size_t(i)], src_ptrs[i], dst_ptrs[i], scratch,
                                  scratch_bytes, stream);
    if (st != RESHARD_OK) return st;
  }
  return RESHARD_OK;
}

reshard_status_t reshard_refit_destroy(reshard_refit_t refit) {
  {
    std::lock_guard<std::mutex> lk(rs::g_refit_mu);
    if (!refit || !rs::refits().erase(refit))
      return fail(RESHARD_ERR_BAD_HANDLE, "refit is NULL or already destroyed");
  }
  if (refit->batch) reshard_batch_destroy(refit->batch);
  delete refit;
  return RESHARD_OK;
}

}  // extern "C"
