// Training-step simulator (DisCo, Simulator): computation operators run one
// at a time from a FIFO ready queue; AllReduce instructions run on one
// channel in the order their (possibly fused) gradient tensors are complete,
// overlapping with computation; an AllReduce of x bytes takes C*x + D
// (DisCo, Profiler).  An operator may also wait for AllReduces (a parameter
// update reading the aggregated gradient): it joins the queue when they are
// scheduled and starts no earlier than their completion.  The result is the
// time the last operator or AllReduce completes.
#include <algorithm>
#include <deque>
#include <queue>
#include <string>
#include <vector>

#include "groupexec.h"

namespace fg {
int set_last_error(int status, const char* msg);
}

namespace {

fg_status bad(const char* msg) { return (fg_status)fg::set_last_error(FG_EINVAL, msg); }

}  // namespace

extern "C" fg_status fg_simulate(const fg_sim_problem* p, double* total, double* op_finish, double* ar_start,
                                 double* ar_finish) {
  if (!p || !total) return bad("null argument");
  const int n = p->n_ops, nb = p->n_buckets, nt = p->n_tensors;
  if (n < 0 || nb < 0 || nt < 0 || p->n_edges < 0 || p->n_ar_edges < 0) return bad("negative count");
  if ((n && !p->op_time) || (p->n_edges && (!p->edge_src || !p->edge_dst)) ||
      (nt && (!p->tensor_producer || !p->tensor_bytes)) || (nb && !p->bucket_bounds) ||
      (p->n_ar_edges && (!p->ar_edge_bucket || !p->ar_edge_op)))
    return bad("null array");
  std::vector<std::vector<int>> succ(n);
  std::vector<int> pending(n, 0);
  for (int e = 0; e < p->n_edges; ++e) {
    const int s = p->edge_src[e], t = p->edge_dst[e];
    if (s < 0 || s >= n || t < 0 || t >= n) return bad("edge out of range");
    succ[s].push_back(t);
    ++pending[t];
  }
  for (int i = 0; i < n; ++i) std::sort(succ[i].begin(), succ[i].end());
  std::vector<std::vector<int>> waits(n), readers(nb);
  for (int e = 0; e < p->n_ar_edges; ++e) {
    const int b = p->ar_edge_bucket[e], t = p->ar_edge_op[e];
    if (b < 0 || b >= nb || t < 0 || t >= n) return bad("AllReduce dependency out of range");
    waits[t].push_back(b);
    readers[b].push_back(t);
    ++pending[t];
  }
  for (int b = 0; b < nb; ++b) std::sort(readers[b].begin(), readers[b].end());
  // per bucket: tensors still to come, bytes; per operator: buckets it feeds
  std::vector<int> left(nb, 0);
  std::vector<double> bytes(nb, 0.0);
  std::vector<std::vector<int>> feeds(n);
  for (int b = 0; b < nb; ++b) {
    if (p->bucket_bounds[b] > p->bucket_bounds[b + 1] || p->bucket_bounds[b] < 0) return bad("bad bucket bounds");
    for (int k = p->bucket_bounds[b]; k < p->bucket_bounds[b + 1]; ++k) {
      const int t = p->bucket_tensors[k];
      if (t < 0 || t >= nt) return bad("bucket tensor out of range");
      const int prod = p->tensor_producer[t];
      if (prod < 0 || prod >= n) return bad("tensor producer out of range");
      ++left[b];
      bytes[b] += p->tensor_bytes[t];
      feeds[prod].push_back(b);
    }
  }

  std::vector<double> fin(n, 0.0), as(nb, -1.0), af(nb, -1.0);
  double device = 0.0, channel = 0.0;
  std::deque<int> queue;
  for (int i = 0; i < n; ++i)
    if (!pending[i]) queue.push_back(i);
  // complete buckets not yet started, by (time complete, bucket)
  using Ev = std::pair<double, int>;
  std::priority_queue<Ev, std::vector<Ev>, std::greater<Ev>> ready_ar;
  auto start_allreduces = [&](double upto) {
    while (!ready_ar.empty() && ready_ar.top().first <= upto) {
      const Ev e = ready_ar.top();
      ready_ar.pop();
      const int b = e.second;
      as[b] = std::max(e.first, channel);
      af[b] = as[b] + p->ar_c * bytes[b] + p->ar_d;
      channel = af[b];
      for (int r : readers[b])
        if (--pending[r] == 0) queue.push_back(r);
    }
  };
  for (int b = 0; b < nb; ++b)
    if (!left[b]) ready_ar.push({0.0, b});
  start_allreduces(0.0);
  int done = 0;
  while (done < n) {
    if (queue.empty()) {
      if (ready_ar.empty()) return bad("dependency cycle, or an operator waits for an AllReduce that never runs");
      start_allreduces(1e300);
      continue;
    }
    const int i = queue.front();
    queue.pop_front();
    double t0 = device;
    // predecessors ran earlier on the same device: only AllReduces can end later
    for (int b : waits[i]) t0 = std::max(t0, af[b]);
    fin[i] = t0 + p->op_time[i];
    device = fin[i];
    ++done;
    for (int b : feeds[i])
      if (--left[b] == 0) ready_ar.push({fin[i], b});
    for (int s : succ[i])
      if (--pending[s] == 0) queue.push_back(s);
    start_allreduces(device);
  }
  start_allreduces(1e300);
  double end = device;
  for (int b = 0; b < nb; ++b) end = std::max(end, af[b]);
  *total = end;
  if (op_finish) std::copy(fin.begin(), fin.end(), op_finish);
  if (ar_start) std::copy(as.begin(), as.end(), ar_start);
  if (ar_finish) std::copy(af.begin(), af.end(), ar_finish);
  return FG_OK;
}
