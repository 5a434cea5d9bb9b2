// refit.cpp -- one call for a whole model's weight refit.  Every plan is routed
// either to the read-once reshard or to gather-and-broadcast (the hybrid split
// of "Integracio es hibrid megoldas a NeMo RL-ben", news.bpdata.com: the
// feed-forward projections through the Reshard collective, small irregular
// weights through gather-and-broadcast); the reshard group can go out as one
// batch launch, or be spread over a few side streams so that the launches of
// small tensors overlap, and the gather-and-broadcast group shares one scratch
// buffer, used tensor after tensor in stream order.
#include <cuda_runtime.h>

#include <algorithm>
#include <array>
#include <map>
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
  // RESHARD_REFIT_LANES: the reshard group as units in issue order (largest
  // first) -- one plan each, or (with RESHARD_REFIT_BATCH too) the plans that one
  // batch launch merges -- with the side stream each unit runs on; fork/join
  // events; the device they belong to.
  struct Unit {
    std::vector<int32_t> plans;
    reshard_batch_t batch = nullptr;  // merged plans: their own batch (one launch)
    int32_t lane = 0;
  };
  std::vector<Unit> units;
  int device = -1;
  cudaEvent_t fork = nullptr;
  std::array<cudaEvent_t, RESHARD_REFIT_NUM_LANES> join = {};
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

// Side streams of each device, created once and shared by every refit on that
// device (in-order streams: executions that share them run one after another on
// each lane).  They live until the process exits, so the per-stream work-queue
// slots of the copy kernels are not used up by refits created and destroyed.
std::mutex g_lane_mu;
std::map<int, std::array<cudaStream_t, RESHARD_REFIT_NUM_LANES>> g_lanes;
// Executions over the side streams are issued one at a time, whichever refit they
// belong to: a lane that joined one caller's CUDA-graph capture must not receive
// another execution's launches until that execution has joined back.
std::mutex g_issue_mu;

reshard_status_t device_lanes(int dev, std::array<cudaStream_t, RESHARD_REFIT_NUM_LANES>* out) {
  std::lock_guard<std::mutex> lk(g_lane_mu);
  auto it = g_lanes.find(dev);
  if (it == g_lanes.end()) {
    std::array<cudaStream_t, RESHARD_REFIT_NUM_LANES> l = {};
    for (int i = 0; i < RESHARD_REFIT_NUM_LANES; ++i) {
      cudaError_t ce = cudaStreamCreateWithFlags(&l[size_t(i)], cudaStreamNonBlocking);
      if (ce != cudaSuccess) {
        for (int j = 0; j < i; ++j) cudaStreamDestroy(l[size_t(j)]);
        return fail(RESHARD_ERR_CUDA, std::string("cudaStreamCreateWithFlags: ") +
                                          cudaGetErrorString(ce));
      }
    }
    it = g_lanes.emplace(dev, l).first;
  }
  *out = it->second;
  return RESHARD_OK;
}

void release_events(reshard_refit_s* R) {
  if (R->fork) cudaEventDestroy(R->fork);
  for (cudaEvent_t& e : R->join)
    if (e) cudaEventDestroy(e);
  R->fork = nullptr;
  R->join = {};
  for (reshard_refit_s::Unit& u : R->units)
    if (u.batch) reshard_batch_destroy(u.batch);
  R->units.clear();
}

// Units and lanes.  With `merge`, the plans that the refit's batch concatenates
// into one launch (a batch class of several plans) form one unit with a batch of
// their own; every other plan is a unit of one.  Lane assignment is longest
// processing time first: units sorted by the bytes the read-once path moves,
// largest first, each to the lane with the fewest bytes so far (ties: the lower
// lane), so the lanes finish close together.  Issue order is the sorted order.
reshard_status_t assign_lanes(reshard_refit_s* R, bool merge) {
  auto bytes = [&](int32_t i) {
    const reshard_stats_t& s = R->plans[size_t(i)]->stats;
    return s.fanout_read_bytes + s.fanout_write_bytes;
  };
  std::vector<char> merged(R->plans.size(), 0);
  if (merge && R->batch) {
    int32_t ncls = 0;
    std::vector<int32_t> cls(R->reshard_idx.size(), -1);
    reshard_status_t st = reshard_batch_classes(R->batch, &ncls, cls.data());
    if (st != RESHARD_OK) return st;
    std::map<int32_t, std::vector<int32_t>> members;
    for (size_t k = 0; k < cls.size(); ++k)
      if (cls[k] >= 0) members[cls[k]].push_back(R->reshard_idx[k]);
    for (auto& cm : members) {
      if (cm.second.size() < 2) continue;
      std::vector<reshard_plan_t> ps;
      for (int32_t i : cm.second) ps.push_back(R->plans[size_t(i)]);
      reshard_refit_s::Unit u;
      u.plans = cm.second;
      st = reshard_batch_create(ps.data(), int32_t(ps.size()), &u.batch);
      if (st != RESHARD_OK) return st;
      R->units.push_back(u);
      for (int32_t i : cm.second) merged[size_t(i)] = 1;
    }
  }
  for (int32_t i : R->reshard_idx) {
    if (merged[size_t(i)]) continue;
    reshard_refit_s::Unit u;
    u.plans.push_back(i);
    R->units.push_back(u);
  }
  auto unit_bytes = [&](const reshard_refit_s::Unit& u) {
    int64_t b = 0;
    for (int32_t i : u.plans) b += bytes(i);
    return b;
  };
  std::stable_sort(R->units.begin(), R->units.end(),
                   [&](const reshard_refit_s::Unit& a, const reshard_refit_s::Unit& b) {
                     return unit_bytes(a) > unit_bytes(b);
                   });
  std::array<int64_t, RESHARD_REFIT_NUM_LANES> load = {};
  for (reshard_refit_s::Unit& u : R->units) {
    size_t best = 0;
    for (size_t l = 1; l < load.size(); ++l)
      if (load[l] < load[best]) best = l;
    load[best] += unit_bytes(u);
    u.lane = int32_t(best);
  }
  cudaError_t ce = cudaGetDevice(&R->device);
  if (ce != cudaSuccess)
    return fail(RESHARD_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(ce));
  std::array<cudaStream_t, RESHARD_REFIT_NUM_LANES> lanes;
  reshard_status_t st = device_lanes(R->device, &lanes);
  if (st != RESHARD_OK) return st;
  ce = cudaEventCreateWithFlags(&R->fork, cudaEventDisableTiming);
  for (cudaEvent_t& e : R->join)
    if (ce == cudaSuccess) ce = cudaEventCreateWithFlags(&e, cudaEventDisableTiming);
  if (ce != cudaSuccess) {
    release_events(R);
    return fail(RESHARD_ERR_CUDA, std::string("cudaEventCreateWithFlags: ") +
                                      cudaGetErrorString(ce));
  }
  return RESHARD_OK;
}

// The reshard group over the side streams: the lanes wait for the caller's stream
// (fork), each plan runs on its lane, and the caller's stream waits for every lane
// (join) -- also after an error, so that what was enqueued stays ordered before
// the caller's later work.
reshard_status_t execute_lanes(reshard_refit_s* R, const void* const* const* src_ptrs,
                               void* const* const* dst_ptrs, void* stream) {
  int dev = -1;
  cudaError_t ce = cudaGetDevice(&dev);
  if (ce != cudaSuccess)
    return fail(RESHARD_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(ce));
  if (dev != R->device)
    return fail(RESHARD_ERR_INVALID_ARG, "the refit's side streams belong to device " +
                                             std::to_string(R->device) + ", current device is " +
                                             std::to_string(dev));
  std::array<cudaStream_t, RESHARD_REFIT_NUM_LANES> lanes;
  reshard_status_t st = device_lanes(dev, &lanes);
  if (st != RESHARD_OK) return st;
  std::lock_guard<std::mutex> lk(g_issue_mu);
  cudaStream_t caller = static_cast<cudaStream_t>(stream);
  // A lane still belongs to a capture that another execution joined it to until
  // that capture ends: refuse to mix this execution into it.
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  unsigned long long cid = 0;
  ce = cudaStreamGetCaptureInfo(caller, &cs, &cid);
  if (ce != cudaSuccess)
    return fail(RESHARD_ERR_CUDA, std::string("cudaStreamGetCaptureInfo: ") + cudaGetErrorString(ce));
  const unsigned long long caller_id = cs == cudaStreamCaptureStatusActive ? cid : 0;
  for (cudaStream_t l : lanes) {
    cudaStreamCaptureStatus ls = cudaStreamCaptureStatusNone;
    unsigned long long lid = 0;
    ce = cudaStreamGetCaptureInfo(l, &ls, &lid);
    if (ce != cudaSuccess)
      return fail(RESHARD_ERR_CUDA, std::string("cudaStreamGetCaptureInfo: ") + cudaGetErrorString(ce));
    if (ls != cudaStreamCaptureStatusNone && (ls != cudaStreamCaptureStatusActive || lid != caller_id))
      return fail(RESHARD_ERR_UNSUPPORTED,
                  "the side streams are taking part in another stream capture until it ends");
  }
  ce = cudaEventRecord(R->fork, caller);
  if (ce != cudaSuccess)
    return fail(RESHARD_ERR_CUDA, std::string("cudaEventRecord: ") + cudaGetErrorString(ce));
  for (cudaStream_t l : lanes) {
    ce = cudaStreamWaitEvent(l, R->fork, 0);
    if (ce != cudaSuccess)
      return fail(RESHARD_ERR_CUDA, std::string("cudaStreamWaitEvent: ") + cudaGetErrorString(ce));
  }
  for (const reshard_refit_s::Unit& u : R->units) {
    cudaStream_t lane = lanes[size_t(u.lane)];
    if (u.batch) {
      std::vector<const void* const*> s;
      std::vector<void* const*> d;
      for (int32_t i : u.plans) {
        s.push_back(src_ptrs[i]);
        d.push_back(dst_ptrs[i]);
      }
      st = reshard_batch_execute(u.batch, s.data(), d.data(), lane);
    } else {
      const int32_t i = u.plans[0];
      st = reshard_execute(R->plans[size_t(i)], src_ptrs[i], dst_ptrs[i], lane);
    }
    if (st != RESHARD_OK) break;
  }
  std::string msg;  // keep the first error's message over the join's
  if (st != RESHARD_OK) msg = reshard_last_error();
  for (size_t l = 0; l < lanes.size(); ++l) {
    ce = cudaEventRecord(R->join[l], lanes[l]);
    if (ce == cudaSuccess) ce = cudaStreamWaitEvent(caller, R->join[l], 0);
    if (ce != cudaSuccess && st == RESHARD_OK)
      return fail(RESHARD_ERR_CUDA, std::string("lane join: ") + cudaGetErrorString(ce));
  }
  if (st != RESHARD_OK) return fail(st, msg);
  return RESHARD_OK;
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
  if ((flags & ~uint32_t(RESHARD_REFIT_BATCH | RESHARD_REFIT_LANES)) != 0)
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
    if ((flags & RESHARD_REFIT_LANES) && !R->reshard_idx.empty()) {
      reshard_status_t st = rs::assign_lanes(R, (flags & RESHARD_REFIT_BATCH) != 0);
      // the units hold what the whole-group batch was needed for
      if (R->batch) reshard_batch_destroy(R->batch);
      R->batch = nullptr;
      if (st != RESHARD_OK) {
        rs::release_events(R);
        delete R;
        return st;
      }
    }
  } catch (const std::bad_alloc&) {
    if (R->batch) reshard_batch_destroy(R->batch);
    rs::release_events(R);
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
  if (refit->fork) {
    st = rs::execute_lanes(refit, src_ptrs, dst_ptrs, stream);
    if (st != RESHARD_OK) return st;
  } else if (refit->batch) {
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
  rs::release_events(refit);
  delete refit;
  return RESHARD_OK;
}

}  // extern "C"
