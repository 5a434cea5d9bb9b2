// partition.cpp -- one reshard split over several GPUs: the multi-GPU exchange.
//
// A partition cuts a plan by destination ownership.  Given the GPU of every
// source and destination rank and the NVLink domain of every GPU, each GPU
// gets the copy programs that fill its own destination ranks and the list of
// messages it sends and receives, following the two-stage transport of the
// Reshard collective write-ups (news.bpdata.com, "A Reshard kollektiv
// kommunikacio": every contribution crosses the network once, the replicas
// are then assembled inside the NVLink domain with a balanced exchange, the two
// stages pipelined; techfeed.io, section on NVIDIA's implementation: incoming
// data spread as evenly as possible over the replicas that hold it):
//   * a region (a destination class x source class intersection) that a GPU
//     needs and also holds in a local source shard is copied locally;
//   * a domain that needs a region held by a source replica inside it gets it
//     from that replica (stage 0, inside the domain), the least-loaded
//     source GPU first;
//   * a domain that needs a region no GPU of it holds receives it ONCE
//     (stage 0, across domains): the sender is the least-loaded GPU holding a
//     source replica, the receiver the least-loaded GPU of the domain that needs
//     it; the receiver then forwards it to the other GPUs of the domain that
//     need it (stage 1, inside the domain);
//   * every GPU writes each region it got to all of its destination replicas
//     of the region's class (the local fan-out).
// Regions that cross GPUs are cut along their outermost dim into `nchunks`
// pieces, piece i in pipeline chunk i (so every link's bytes split evenly over
// the chunks); chunks alternate between two slots of the send and
// receive buffers, so stage 1 of one chunk can run while stage 0 of the next
// one is in flight.  Messages are packed: all pieces from one GPU to another in
// one chunk and stage are one contiguous range of the sender's send buffer and
// of the receiver's receive buffer, in piece order, each piece 16-byte aligned.
//
// The library moves no bytes between GPUs: the caller performs the messages
// (NCCL point-to-point, peer copies) between the steps that it launches here.
#include <cuda_runtime.h>

#include <algorithm>
#include <chrono>
#include <map>
#include <memory>
#include <mutex>
#include <new>
#include <string>
#include <unordered_set>
#include <vector>

#include "internal.h"

namespace rs {
namespace {

constexpr uint64_t kPartitionMagic = 0x5245534850415254ull;  // "RESHPART"
constexpr int64_t kPieceAlign = 16;
constexpr int32_t kMaxChunks = 64;
constexpr int32_t kMaxGpus = 4096;

int64_t align_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

// A region, or a piece of one, in global coordinates.
struct Piece {
  int64_t lo[RESHARD_MAX_TENSOR_NDIM], ext[RESHARD_MAX_TENSOR_NDIM];
  int64_t bytes = 0;
  size_t d = 0, s = 0;  // destination and source class
  int32_t chunk = 0;
};

// All pieces from one GPU to another in one chunk and stage.
struct Msg {
  int32_t chunk, stage, from, to;
  std::vector<size_t> pieces;   // piece indices, ascending
  std::vector<int64_t> at;      // byte offset of each piece inside the message
  int64_t bytes = 0;            // with the alignment padding
  int64_t send_off = 0, recv_off = 0;
};

struct GpuPart {
  // program holders: [0] LOCAL, then per chunk c: [1 + 3c] PACK, [2 + 3c] FORWARD,
  // [3 + 3c] UNPACK; each keeps its program in prog[RESHARD_PROGRAM_FANOUT]
  std::vector<std::unique_ptr<reshard_plan_s>> holders;
  std::vector<reshard_xfer_t> xfers;
  reshard_partition_gpu_t info = {};
};

}  // namespace
}  // namespace rs

struct reshard_partition_s {
  uint64_t magic = 0;
  int32_t ngpus = 0, nchunks = 1, nslots = 1, ndomains = 0;
  int64_t M = 0, N = 0;
  std::vector<int32_t> src_gpu, dst_gpu;  // -1 for ranks the plan leaves out
  std::vector<std::unique_ptr<rs::GpuPart>> gpu;
  reshard_partition_stats_t stats = {};
  // which source / destination ranks must have a buffer on their GPU
  std::vector<uint8_t> src_needed, dst_needed;
};

namespace rs {
namespace {

std::mutex g_part_mu;
std::unordered_set<const reshard_partition_s*>& partitions() {
  static std::unordered_set<const reshard_partition_s*> p;
  return p;
}
bool part_live(const reshard_partition_s* p) {
  if (!p) return false;
  std::lock_guard<std::mutex> lk(g_part_mu);
  return partitions().count(p) != 0;
}

int holder_index(int32_t step, int32_t chunk) {
  return step == RESHARD_STEP_LOCAL ? 0 : 1 + 3 * chunk + (step - RESHARD_STEP_PACK);
}

// Fan-out groups of buffer indices (at most kMaxGroup each), appended to P.
std::vector<uint16_t> add_groups(Program& P, const std::vector<uint16_t>& bufs) {
  std::vector<uint16_t> ids;
  for (size_t a = 0; a < bufs.size(); a += kMaxGroup) {
    ids.push_back(uint16_t(P.goff.size() - 1));
    for (size_t b = a; b < std::min(bufs.size(), a + size_t(kMaxGroup)); ++b)
      P.gbuf.push_back(bufs[b]);
    P.goff.push_back(uint32_t(P.gbuf.size()));
  }
  return ids;
}

// Least-loaded candidate (ties: lowest index).
int32_t least(const std::vector<int32_t>& cands, const std::vector<int64_t>& load) {
  int32_t best = -1;
  for (int32_t g : cands)
    if (best < 0 || load[size_t(g)] < load[size_t(best)]) best = g;
  return best;
}

reshard_status_t build_partition(const reshard_plan_s* P, reshard_partition_s* X,
                                 const int32_t* gpu_domain) {
  const int32_t nd = P->ndim;
  const int64_t eb = P->elem_bytes;
  const int64_t M = P->src.nranks, N = P->dst.nranks;
  const int32_t G = X->ngpus, C = X->nchunks;
  const uint16_t recv_buf = uint16_t(M + N), send_buf = uint16_t(M + N + 1);
  const std::vector<Class> sc = classes_of(nd, P->src, P->src_gone);
  const std::vector<Class> dc = classes_of(nd, P->dst, P->dst_gone);
  reshard_partition_stats_t& S = X->stats;
  X->src_needed.assign(size_t(M), 0);
  X->dst_needed.assign(size_t(N), 0);

  // GPUs holding each class's ranks, ascending
  auto gpus_of = [&](const Class& c, const std::vector<int32_t>& where) {
    std::vector<int32_t> g;
    for (int64_t r : c.ranks) g.push_back(where[size_t(r)]);
    std::sort(g.begin(), g.end());
    g.erase(std::unique(g.begin(), g.end()), g.end());
    return g;
  };
  std::vector<std::vector<int32_t>> src_gpus(sc.size()), dst_gpus(dc.size());
  for (size_t i = 0; i < sc.size(); ++i) src_gpus[i] = gpus_of(sc[i], X->src_gpu);
  for (size_t i = 0; i < dc.size(); ++i) dst_gpus[i] = gpus_of(dc[i], X->dst_gpu);
  for (const Class& c : dc)
    for (int64_t r : c.ranks) X->dst_needed[size_t(r)] = 1;

  // intersections; the ones some GPU needs from another GPU become pieces
  struct Local {
    Piece g;
    int64_t src_rank;
    int32_t gpu;
  };
  std::vector<Local> locals;
  std::vector<Piece> pieces;
  int64_t rotate = 0;
  for (size_t di = 0; di < dc.size(); ++di) {
    for (size_t si = 0; si < sc.size(); ++si) {
      Piece g;
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
      bool remote = false;
      for (int32_t gpu : dst_gpus[di]) {
        int64_t here = -1;
        for (int64_t r : sc[si].ranks)
          if (X->src_gpu[size_t(r)] == gpu) {
            here = r;
            break;
          }
        if (here >= 0) {
          locals.push_back({g, here, gpu});
          X->src_needed[size_t(here)] = 1;
        } else {
          remote = true;
        }
      }
      if (!remote) continue;
      // cut along the outermost dim of extent > 1 into C pieces, piece i into chunk i,
      // so that every link's bytes split evenly over the chunks; a region with fewer
      // rows than chunks gives one piece per row, to chunks taken in turn
      int cut = -1;
      for (int d = 0; d < nd && cut < 0; ++d)
        if (g.ext[d] > 1) cut = d;
      const int64_t k = cut < 0 ? 1 : std::min<int64_t>(C, g.ext[cut]);
      for (int64_t i = 0; i < k; ++i) {
        Piece q = g;
        if (cut >= 0) {
          const int64_t a = g.ext[cut] * i / k, b = g.ext[cut] * (i + 1) / k;
          q.lo[cut] = g.lo[cut] + a;
          q.ext[cut] = b - a;
          q.bytes = g.bytes / g.ext[cut] * (b - a);
        }
        q.chunk = int32_t((rotate + i) % C);
        pieces.push_back(q);
      }
      // the next region starts its pieces one chunk later (k == C: the larger pieces
      // of uneven cuts spread over the chunks) or after this one's (k < C)
      rotate = (rotate + (k < C ? k : 1)) % C;
    }
  }
  std::vector<size_t> order(pieces.size());
  for (size_t i = 0; i < order.size(); ++i) order[i] = i;
  std::stable_sort(order.begin(), order.end(),
                   [&](size_t a, size_t b) { return pieces[a].bytes > pieces[b].bytes; });

  // senders and receivers, largest piece first onto the least-loaded GPU
  std::map<std::vector<int32_t>, size_t> msg_index;  // (chunk, stage, from, to)
  std::vector<Msg> msgs;
  auto add = [&](size_t pi, int32_t stage, int32_t from, int32_t to) {
    const std::vector<int32_t> key = {pieces[pi].chunk, stage, from, to};
    auto it = msg_index.find(key);
    if (it == msg_index.end()) {
      it = msg_index.emplace(key, msgs.size()).first;
      msgs.push_back(Msg{pieces[pi].chunk, stage, from, to, {}, {}, 0, 0, 0});
    }
    msgs[it->second].pieces.push_back(pi);
    const bool across = gpu_domain[from] != gpu_domain[to];
    (across ? S.inter_domain_bytes : S.intra_domain_bytes) += pieces[pi].bytes;
    (across ? X->gpu[size_t(from)]->info.sent_inter_bytes
            : X->gpu[size_t(from)]->info.sent_intra_bytes) += pieces[pi].bytes;
    (across ? X->gpu[size_t(to)]->info.recv_inter_bytes
            : X->gpu[size_t(to)]->info.recv_intra_bytes) += pieces[pi].bytes;
  };
  std::vector<int64_t> send0(size_t(G), 0), recv0(size_t(G), 0);
  for (size_t pi : order) {
    const Piece& g = pieces[pi];
    const std::vector<int32_t>& have = src_gpus[g.s];
    std::map<int32_t, std::vector<int32_t>> by_domain;  // domain -> GPUs without a source
    for (int32_t gpu : dst_gpus[g.d])
      if (!std::binary_search(have.begin(), have.end(), gpu))
        by_domain[gpu_domain[gpu]].push_back(gpu);
    for (const auto& kv : by_domain) {
      std::vector<int32_t> inside;
      for (int32_t h : have)
        if (gpu_domain[h] == kv.first) inside.push_back(h);
      if (!inside.empty()) {
        for (int32_t to : kv.second) {
          const int32_t from = least(inside, send0);
          send0[size_t(from)] += g.bytes;
          add(pi, 0, from, to);
        }
        continue;
      }
      const int32_t from = least(have, send0);
      const int32_t recv = least(kv.second, recv0);
      send0[size_t(from)] += g.bytes;
      recv0[size_t(recv)] += g.bytes;
      add(pi, 0, from, recv);
      for (int32_t to : kv.second)
        if (to != recv) add(pi, 1, recv, to);
    }
  }

  // message layout: per GPU and chunk, stage 0 then stage 1, peers ascending
  std::sort(msgs.begin(), msgs.end(), [](const Msg& a, const Msg& b) {
    if (a.chunk != b.chunk) return a.chunk < b.chunk;
    if (a.stage != b.stage) return a.stage < b.stage;
    if (a.from != b.from) return a.from < b.from;
    return a.to < b.to;
  });
  for (Msg& m : msgs) {
    std::sort(m.pieces.begin(), m.pieces.end());
    for (size_t pi : m.pieces) {
      m.at.push_back(m.bytes);
      m.bytes = align_up(m.bytes + pieces[pi].bytes, kPieceAlign);
    }
  }
  // bytes of each (GPU, chunk) on the send and the receive side; a slot holds the largest
  std::vector<int64_t> send_cur(size_t(G) * size_t(C), 0), recv_cur(size_t(G) * size_t(C), 0);
  for (Msg& m : msgs) {
    int64_t& so = send_cur[size_t(m.from) * size_t(C) + size_t(m.chunk)];
    int64_t& ro = recv_cur[size_t(m.to) * size_t(C) + size_t(m.chunk)];
    m.send_off = so;  // relative to the chunk's slot for now
    m.recv_off = ro;
    so += m.bytes;
    ro += m.bytes;
  }
  std::vector<int64_t> send_slot(size_t(G), 0), recv_slot(size_t(G), 0);
  for (int32_t g = 0; g < G; ++g)
    for (int32_t c = 0; c < C; ++c) {
      send_slot[size_t(g)] = std::max(send_slot[size_t(g)], send_cur[size_t(g) * C + c]);
      recv_slot[size_t(g)] = std::max(recv_slot[size_t(g)], recv_cur[size_t(g) * C + c]);
    }
  for (Msg& m : msgs) {
    m.send_off += int64_t(m.chunk % X->nslots) * send_slot[size_t(m.from)];
    m.recv_off += int64_t(m.chunk % X->nslots) * recv_slot[size_t(m.to)];
  }
  // where each piece landed at each GPU in stage 0 (the forwarding source)
  std::map<std::pair<size_t, int32_t>, int64_t> landed;
  for (const Msg& m : msgs)
    if (m.stage == 0)
      for (size_t k = 0; k < m.pieces.size(); ++k)
        landed[{m.pieces[k], m.to}] = m.recv_off + m.at[k];

  // programs
  for (int32_t g = 0; g < G; ++g) {
    GpuPart& part = *X->gpu[size_t(g)];
    part.holders.resize(size_t(1 + 3 * C));
    for (auto& h : part.holders) {
      h.reset(new reshard_plan_s());
      for (int k = 0; k < kNumPrograms; ++k) h->prog[k].goff.push_back(0);
      h->ndim = nd;
      h->elem_bytes = int32_t(eb);
    }
    part.info.send_bytes = int64_t(X->nslots) * send_slot[size_t(g)];
    part.info.recv_bytes = int64_t(X->nslots) * recv_slot[size_t(g)];
  }
  auto prog_of = [&](int32_t g, int32_t step, int32_t chunk) -> Program& {
    return X->gpu[size_t(g)]->holders[size_t(holder_index(step, chunk))]->prog[RESHARD_PROGRAM_FANOUT];
  };
  // destination buffers of a class on one GPU
  auto local_dsts = [&](size_t di, int32_t g) {
    std::vector<uint16_t> b;
    for (int64_t r : dc[di].ranks)
      if (X->dst_gpu[size_t(r)] == g) b.push_back(uint16_t(M + r));
    return b;
  };
  auto box_place = [&](const Piece& q, const Box& side, int64_t* st) {
    row_major_strides(nd, side.shp, st);
    int64_t o = 0;
    for (int d = 0; d < nd; ++d) o += (q.lo[d] - side.off[d]) * st[d];
    return o;
  };
  // LOCAL: source shard on the GPU -> its destination replicas of the class
  for (const Local& l : locals) {
    Program& PL = prog_of(l.gpu, RESHARD_STEP_LOCAL, 0);
    const std::vector<uint16_t> dsts = local_dsts(l.g.d, l.gpu);
    int64_t sst[RESHARD_MAX_TENSOR_NDIM], dst[RESHARD_MAX_TENSOR_NDIM];
    const int64_t s0 = box_place(l.g, P->src.box[size_t(l.src_rank)], sst);
    const int64_t d0 = box_place(l.g, dc[l.g.d].box, dst);
    for (uint16_t grp : add_groups(PL, dsts))
      emit_box(PL, uint16_t(l.src_rank), grp, nd, l.g.ext, s0, sst, d0, dst, eb,
               int64_t(PL.goff[grp + 1] - PL.goff[grp]));
    X->gpu[size_t(l.gpu)]->info.local_bytes += l.g.bytes;
    S.local_bytes += l.g.bytes * int64_t(dsts.size());
  }
  for (const Msg& m : msgs) {
    for (size_t k = 0; k < m.pieces.size(); ++k) {
      const Piece& q = pieces[m.pieces[k]];
      int64_t pst[RESHARD_MAX_TENSOR_NDIM];
      row_major_strides(nd, q.ext, pst);  // packed layout of the piece
      // sender: PACK from a source shard (stage 0) or FORWARD what it received (stage 1)
      if (m.stage == 0) {
        Program& PP = prog_of(m.from, RESHARD_STEP_PACK, m.chunk);
        int64_t rank = -1;
        for (int64_t r : sc[q.s].ranks)
          if (X->src_gpu[size_t(r)] == m.from) {
            rank = r;
            break;
          }
        X->src_needed[size_t(rank)] = 1;
        int64_t sst[RESHARD_MAX_TENSOR_NDIM];
        const int64_t s0 = box_place(q, P->src.box[size_t(rank)], sst);
        const uint16_t grp = add_groups(PP, {send_buf})[0];
        emit_box(PP, uint16_t(rank), grp, nd, q.ext, s0, sst, (m.send_off + m.at[k]) / eb, pst,
                 eb);
      } else {
        Program& PF = prog_of(m.from, RESHARD_STEP_FORWARD, m.chunk);
        const int64_t from_off = landed.at({m.pieces[k], m.from});
        const int64_t n = q.bytes / eb, one = 1;
        const uint16_t grp = add_groups(PF, {send_buf})[0];
        emit_box(PF, recv_buf, grp, 1, &n, from_off / eb, &one, (m.send_off + m.at[k]) / eb,
                 &one, eb);
      }
      // receiver: UNPACK into its destination replicas of the class
      Program& PU = prog_of(m.to, RESHARD_STEP_UNPACK, m.chunk);
      int64_t dst[RESHARD_MAX_TENSOR_NDIM];
      const int64_t d0 = box_place(q, dc[q.d].box, dst);
      for (uint16_t grp : add_groups(PU, local_dsts(q.d, m.to)))
        emit_box(PU, recv_buf, grp, nd, q.ext, (m.recv_off + m.at[k]) / eb, pst, d0, dst, eb,
                 int64_t(PU.goff[grp + 1] - PU.goff[grp]));
    }
    GpuPart& from = *X->gpu[size_t(m.from)];
    GpuPart& to = *X->gpu[size_t(m.to)];
    from.xfers.push_back({m.chunk, m.stage, m.to, 0, m.send_off, m.bytes});
    to.xfers.push_back({m.chunk, m.stage, m.from, 1, m.recv_off, m.bytes});
  }
  for (int32_t g = 0; g < G; ++g) {
    GpuPart& part = *X->gpu[size_t(g)];
    for (auto& h : part.holders) {
      Program& p = h->prog[RESHARD_PROGRAM_FANOUT];
      if (p.goff.size() > 65536) return fail(RESHARD_ERR_UNSUPPORTED, "more than 65535 groups");
      finish_program(p);
      p.staged = true;
      for (int k = 0; k < kNumPrograms; ++k)
        if (k != RESHARD_PROGRAM_FANOUT) finish_program(h->prog[k]);
    }
    std::sort(part.xfers.begin(), part.xfers.end(),
              [](const reshard_xfer_t& a, const reshard_xfer_t& b) {
                if (a.chunk != b.chunk) return a.chunk < b.chunk;
                if (a.stage != b.stage) return a.stage < b.stage;
                if (a.dir != b.dir) return a.dir < b.dir;
                return a.peer < b.peer;
              });
    part.info.n_xfers = int64_t(part.xfers.size());
    S.max_gpu_send_bytes = std::max(S.max_gpu_send_bytes,
                                    part.info.sent_inter_bytes + part.info.sent_intra_bytes);
    S.max_gpu_recv_bytes = std::max(S.max_gpu_recv_bytes,
                                    part.info.recv_inter_bytes + part.info.recv_intra_bytes);
  }
  S.n_pieces = int64_t(pieces.size());
  S.n_messages = int64_t(msgs.size());
  return RESHARD_OK;
}

void free_partition(reshard_partition_s* X) {
  for (auto& part : X->gpu) {
    if (!part) continue;
    for (auto& h : part->holders) {
      if (!h || !h->d_mem) continue;
      int cur = -1;
      cudaGetDevice(&cur);
      if (cur != h->device) cudaSetDevice(h->device);
      cudaFree(h->d_mem);
      h->d_mem = nullptr;
      if (cur >= 0 && cur != h->device) cudaSetDevice(cur);
    }
  }
  X->magic = 0;
  delete X;
}

reshard_status_t check_step(const reshard_partition_s* X, int32_t gpu, int32_t step,
                            int32_t chunk) {
  if (!part_live(X)) return fail(RESHARD_ERR_BAD_HANDLE, "invalid partition handle");
  if (gpu < 0 || gpu >= X->ngpus) return fail(RESHARD_ERR_INVALID_ARG, "gpu out of range");
  if (step < RESHARD_STEP_LOCAL || step > RESHARD_STEP_UNPACK)
    return fail(RESHARD_ERR_INVALID_ARG, "unknown step");
  if (step != RESHARD_STEP_LOCAL && (chunk < 0 || chunk >= X->nchunks))
    return fail(RESHARD_ERR_INVALID_ARG, "chunk out of range");
  return RESHARD_OK;
}

}  // namespace
}  // namespace rs

using rs::fail;

extern "C" {

reshard_status_t reshard_partition_create(reshard_plan_t plan, const int32_t* src_gpu,
                                          const int32_t* dst_gpu, int32_t ngpus,
                                          const int32_t* gpu_domain, int32_t nchunks,
                                          reshard_partition_t* out_partition) {
  const auto t0 = std::chrono::steady_clock::now();
  rs::TraceRange trace("reshard.partition");
  if (!out_partition) return fail(RESHARD_ERR_INVALID_ARG, "out_partition is NULL");
  *out_partition = nullptr;
  if (!rs::plan_live(plan)) return fail(RESHARD_ERR_BAD_HANDLE, "invalid plan handle");
  if (plan->inplace) return fail(RESHARD_ERR_UNSUPPORTED, "in-place plans cannot be partitioned");
  if (ngpus < 1 || ngpus > rs::kMaxGpus) return fail(RESHARD_ERR_INVALID_ARG, "ngpus must be 1..4096");
  if (nchunks < 1 || nchunks > rs::kMaxChunks)
    return fail(RESHARD_ERR_INVALID_ARG, "nchunks must be 1..64");
  if (!src_gpu || !dst_gpu || !gpu_domain) return fail(RESHARD_ERR_INVALID_ARG, "null map");
  const int64_t M = plan->src.nranks, N = plan->dst.nranks;
  if (M + N + 2 > RESHARD_MAX_EXEC_BUFFERS)
    return fail(RESHARD_ERR_UNSUPPORTED, "M + N + 2 exceeds RESHARD_MAX_EXEC_BUFFERS");
  for (int32_t g = 0; g < ngpus; ++g)
    if (gpu_domain[g] < 0) return fail(RESHARD_ERR_INVALID_ARG, "negative domain");
  auto gone = [](const std::vector<uint8_t>& v, int64_t r) { return !v.empty() && v[size_t(r)]; };
  for (int64_t r = 0; r < M; ++r)
    if (!gone(plan->src_gone, r) && (src_gpu[r] < 0 || src_gpu[r] >= ngpus))
      return fail(RESHARD_ERR_INVALID_ARG, "source rank " + std::to_string(r) + ": gpu out of range");
  for (int64_t r = 0; r < N; ++r)
    if (!gone(plan->dst_gone, r) && (dst_gpu[r] < 0 || dst_gpu[r] >= ngpus))
      return fail(RESHARD_ERR_INVALID_ARG,
                  "destination rank " + std::to_string(r) + ": gpu out of range");
  reshard_partition_s* X = new (std::nothrow) reshard_partition_s();
  if (!X) return fail(RESHARD_ERR_NO_MEMORY, "host allocation failed");
  reshard_status_t st = RESHARD_OK;
  try {
    X->ngpus = ngpus;
    X->nchunks = nchunks;
    X->nslots = nchunks > 1 ? 2 : 1;
    X->M = M;
    X->N = N;
    X->src_gpu.assign(src_gpu, src_gpu + M);
    X->dst_gpu.assign(dst_gpu, dst_gpu + N);
    for (int64_t r = 0; r < M; ++r)
      if (gone(plan->src_gone, r)) X->src_gpu[size_t(r)] = -1;
    for (int64_t r = 0; r < N; ++r)
      if (gone(plan->dst_gone, r)) X->dst_gpu[size_t(r)] = -1;
    std::vector<int32_t> doms(gpu_domain, gpu_domain + ngpus);
    std::sort(doms.begin(), doms.end());
    X->ndomains = int32_t(std::unique(doms.begin(), doms.end()) - doms.begin());
    X->gpu.resize(size_t(ngpus));
    for (auto& g : X->gpu) g.reset(new rs::GpuPart());
    st = rs::build_partition(plan, X, gpu_domain);
  } catch (const std::bad_alloc&) {
    st = fail(RESHARD_ERR_NO_MEMORY, "host allocation failed while partitioning");
  }
  if (st != RESHARD_OK) {
    rs::free_partition(X);
    return st;
  }
  X->stats.ngpus = ngpus;
  X->stats.ndomains = X->ndomains;
  X->stats.nchunks = nchunks;
  X->stats.nslots = X->nslots;
  X->stats.planner_ns = std::chrono::duration_cast<std::chrono::nanoseconds>(
                            std::chrono::steady_clock::now() - t0).count();
  X->magic = rs::kPartitionMagic;
  {
    std::lock_guard<std::mutex> lk(rs::g_part_mu);
    rs::partitions().insert(X);
  }
  *out_partition = X;
  return RESHARD_OK;
}

reshard_status_t reshard_partition_stats(reshard_partition_t part, reshard_partition_stats_t* out) {
  if (!rs::part_live(part)) return fail(RESHARD_ERR_BAD_HANDLE, "invalid partition handle");
  if (!out) return fail(RESHARD_ERR_INVALID_ARG, "out is NULL");
  *out = part->stats;
  return RESHARD_OK;
}

reshard_status_t reshard_partition_gpu(reshard_partition_t part, int32_t gpu,
                                       reshard_partition_gpu_t* out) {
  reshard_status_t st = rs::check_step(part, gpu, RESHARD_STEP_LOCAL, 0);
  if (st != RESHARD_OK) return st;
  if (!out) return fail(RESHARD_ERR_INVALID_ARG, "out is NULL");
  *out = part->gpu[size_t(gpu)]->info;
  return RESHARD_OK;
}

reshard_status_t reshard_partition_transfers(reshard_partition_t part, int32_t gpu,
                                             const reshard_xfer_t** xfers, int64_t* n) {
  reshard_status_t st = rs::check_step(part, gpu, RESHARD_STEP_LOCAL, 0);
  if (st != RESHARD_OK) return st;
  if (!xfers || !n) return fail(RESHARD_ERR_INVALID_ARG, "null output");
  *xfers = part->gpu[size_t(gpu)]->xfers.data();
  *n = int64_t(part->gpu[size_t(gpu)]->xfers.size());
  return RESHARD_OK;
}

reshard_status_t reshard_partition_program(reshard_partition_t part, int32_t gpu, int32_t step,
                                           int32_t chunk, const reshard_tile_t** tiles,
                                           int64_t* ntiles, const int64_t** unit_prefix,
                                           const uint32_t** group_offsets,
                                           const uint16_t** group_buffers, int64_t* ngroups) {
  reshard_status_t st = rs::check_step(part, gpu, step, chunk);
  if (st != RESHARD_OK) return st;
  const rs::Program& p = part->gpu[size_t(gpu)]
                             ->holders[size_t(rs::holder_index(step, chunk))]
                             ->prog[RESHARD_PROGRAM_FANOUT];
  if (tiles) *tiles = p.tiles.data();
  if (ntiles) *ntiles = int64_t(p.tiles.size());
  if (unit_prefix) *unit_prefix = p.prefix.data();
  if (group_offsets) *group_offsets = p.goff.data();
  if (group_buffers) *group_buffers = p.gbuf.data();
  if (ngroups) *ngroups = int64_t(p.goff.size()) - 1;
  return RESHARD_OK;
}

reshard_status_t reshard_partition_execute(reshard_partition_t part, int32_t gpu, int32_t step,
                                           int32_t chunk, const void* const* src_ptrs,
                                           void* const* dst_ptrs, void* recv_buf, void* send_buf,
                                           void* stream) {
  rs::TraceRange trace("reshard.partition_exec");
  reshard_status_t st = rs::check_step(part, gpu, step, chunk);
  if (st != RESHARD_OK) return st;
  if (!src_ptrs || !dst_ptrs) return fail(RESHARD_ERR_INVALID_ARG, "null pointer array");
  const int64_t M = part->M, N = part->N;
  const rs::GpuPart& gp = *part->gpu[size_t(gpu)];
  if (gp.info.recv_bytes > 0 && !recv_buf)
    return fail(RESHARD_ERR_INVALID_ARG, "recv_buf is NULL");
  if (gp.info.send_bytes > 0 && !send_buf)
    return fail(RESHARD_ERR_INVALID_ARG, "send_buf is NULL");
  // buffer table [sources..., destinations..., receive, send]; ranks on other GPUs
  // are never addressed and enter the table as NULL
  unsigned char* bufs[RESHARD_MAX_EXEC_BUFFERS];
  for (int64_t r = 0; r < M; ++r) {
    const bool here = part->src_gpu[size_t(r)] == gpu;
    if (here && part->src_needed[size_t(r)] && !src_ptrs[r])
      return fail(RESHARD_ERR_INVALID_ARG,
                  "NULL source pointer for source rank " + std::to_string(r) + " on this gpu");
    bufs[r] = here ? static_cast<unsigned char*>(const_cast<void*>(src_ptrs[r])) : nullptr;
  }
  for (int64_t r = 0; r < N; ++r) {
    const bool here = part->dst_gpu[size_t(r)] == gpu;
    if (here && part->dst_needed[size_t(r)] && !dst_ptrs[r])
      return fail(RESHARD_ERR_INVALID_ARG, "NULL destination pointer for destination rank " +
                                               std::to_string(r) + " on this gpu");
    bufs[M + r] = here ? static_cast<unsigned char*>(dst_ptrs[r]) : nullptr;
  }
  bufs[M + N] = static_cast<unsigned char*>(recv_buf);
  bufs[M + N + 1] = static_cast<unsigned char*>(send_buf);
  reshard_plan_s* h = gp.holders[size_t(rs::holder_index(step, chunk))].get();
  if (h->prog[RESHARD_PROGRAM_FANOUT].total_units() == 0) return RESHARD_OK;
  st = rs::upload_plan(h);
  if (st != RESHARD_OK) return st;
  return rs::launch_program(h, h->prog[RESHARD_PROGRAM_FANOUT], bufs, int(M + N + 2), stream);
}

reshard_status_t reshard_partition_destroy(reshard_partition_t part) {
  {
    std::lock_guard<std::mutex> lk(rs::g_part_mu);
    if (!part || !rs::partitions().erase(part))
      return fail(RESHARD_ERR_BAD_HANDLE, "partition is NULL or already destroyed");
  }
  rs::free_partition(part);
  return RESHARD_OK;
}

}  // extern "C"
