// Host-side DASH schedule tables and the compute/reduce DAG simulator.
//
// Task orders ("DASH: Deterministic Attention Scheduling for High-throughput Reproducible
// LLM Training": abstract; Pith review "What carries the argument"; Figure 3, 4, 6, 7):
//   ascending        KV_i visits its Q tiles upwards (FlashAttention-3 baseline)
//   descending       KV_i visits its Q tiles downwards (Descending Q-Tile Iteration)
//   shift            full mask: step t of KV_i works on Q_((i+t) mod n)
//   symmetric shift  causal, n even: slot p runs KV_p over the lower-left rectangle with
//                    a cyclic shift, then KV_p's upper-left triangle upwards from the
//                    diagonal, then KV_(n-1-p)'s lower-right triangle downwards.
// dQ_j reduction order: ascending KV index for ascending/descending; the arrival step
// (position in the chain) for shift and symmetric shift, which never puts two chains
// on one dQ block at the same step. On a persistent grid that runs a head's chains in
// more than one round, shift and symmetric shift order by arrival under the dealing
// (dealt_orders below).
#include "sched.h"

#include <algorithm>
#include <functional>
#include <queue>

namespace dash {

namespace {
inline int32_t pack(int kv, int q) { return (int32_t)((kv << 16) | q); }
}  // namespace

int build_schedule(int mask, int sched, int n, Schedule* out) {
  if (n < 1 || n > 32767) return 1;                         // DASH_ERR_INVALID_ARG
  if (mask != MASK_FULL && mask != MASK_CAUSAL) return 1;
  if (sched < SCHED_ASCENDING || sched > SCHED_SYMMETRIC_SHIFT) return 1;
  if (sched == SCHED_SHIFT && mask != MASK_FULL) return 2;  // DASH_ERR_UNSUPPORTED
  if (sched == SCHED_SYMMETRIC_SHIFT && (mask != MASK_CAUSAL || (n & 1))) return 2;

  Schedule s;
  s.mask = mask;
  s.sched = sched;
  s.n = n;
  const bool causal = mask == MASK_CAUSAL;
  std::vector<std::vector<int32_t>> chains;
  if (sched == SCHED_SYMMETRIC_SHIFT) {
    const int half = n / 2;
    for (int p = 0; p < half; ++p) {
      std::vector<int32_t> ch;
      for (int t = 0; t < half; ++t) ch.push_back(pack(p, half + (p + t) % half));
      for (int u = 0; u < half - p; ++u) ch.push_back(pack(p, p + u));
      for (int u = 0; u <= p; ++u) ch.push_back(pack(n - 1 - p, n - 1 - u));
      chains.push_back(std::move(ch));
    }
  } else {
    for (int i = 0; i < n; ++i) {
      std::vector<int32_t> ch;
      const int lo = causal ? i : 0;
      const int len = n - lo;
      for (int t = 0; t < len; ++t) {
        int q;
        if (sched == SCHED_ASCENDING) q = lo + t;
        else if (sched == SCHED_DESCENDING) q = n - 1 - t;
        else q = (i + t) % n;                                  // shift (full only)
        ch.push_back(pack(i, q));
      }
      chains.push_back(std::move(ch));
    }
  }
  s.num_slots = (int)chains.size();
  s.slot_off.assign(s.num_slots + 1, 0);
  for (int p = 0; p < s.num_slots; ++p) {
    s.slot_off[p + 1] = s.slot_off[p] + (int32_t)chains[p].size();
    s.max_chain = std::max(s.max_chain, (int)chains[p].size());
    s.tasks.insert(s.tasks.end(), chains[p].begin(), chains[p].end());
  }

  // Reduction order per dQ block.
  s.ord.assign((size_t)n * n, -1);
  s.cnt.assign(n, 0);
  if (sched == SCHED_ASCENDING || sched == SCHED_DESCENDING) {
    for (int j = 0; j < n; ++j) {
      int k = 0;
      for (int i = 0; i < n; ++i)
        if (!causal || j >= i) s.ord[(size_t)i * n + j] = k++;
      s.cnt[j] = k;
    }
  } else {
    // arrival step; no two chains share (step, q tile) -- checked here
    std::vector<std::vector<std::pair<int, int>>> arrivals(n);  // (step, kv)
    for (int p = 0; p < s.num_slots; ++p)
      for (int t = 0; t < (int)chains[p].size(); ++t) {
        const int kv = chains[p][t] >> 16, q = chains[p][t] & 0xffff;
        arrivals[q].push_back({t, kv});
      }
    for (int j = 0; j < n; ++j) {
      auto& a = arrivals[j];
      std::sort(a.begin(), a.end());
      for (size_t k = 0; k < a.size(); ++k) {
        if (k && a[k].first == a[k - 1].first) return 2;        // conflicting step
        s.ord[(size_t)a[k].second * n + j] = (int32_t)k;
      }
      s.cnt[j] = (int)a.size();
    }
  }
  *out = std::move(s);
  return 0;
}

void deal(const Schedule& sc, int heads, int grid, int head_dim, Dealing* out) {
  out->cta_off.assign(grid + 1, 0);
  out->pieces.clear();
  const long long units = (long long)heads * sc.num_slots;
  const long long rem = units % grid;
  std::vector<std::vector<Piece>> per_cta(grid);
  auto unit_piece = [&](long long u) {
    const int slot = (int)(u % sc.num_slots);
    Piece pc;
    pc.head = (int32_t)(u / sc.num_slots);
    pc.t_begin = sc.slot_off[slot];
    pc.t_end = sc.slot_off[slot + 1];
    return pc;
  };
  if (!arrival_ordered(sc) || rem == 0 || units < grid) {
    // round robin: unit u = (head u / slots, slot u % slots) to CTA u % grid
    for (long long u = 0; u < units; ++u) per_cta[u % grid].push_back(unit_piece(u));
  } else if (sc.sched == SCHED_SHIFT) {
    // one KV tile per unit, all of one length: round robin, with the last partial round's
    // tiles halved over two CTAs where there is room
    // (Holding back the highest slots of every head instead, so that the halves spread
    // over the heads, measured slower in deterministic mode on GB300: it lengthens the
    // turn waits of the earlier rounds more than the last head's denser dQ order costs.)
    const long long splits = split_tiles(sc.sched, sc.n, units, grid);
    const long long whole = units - splits;
    for (long long u = 0; u < whole; ++u) per_cta[u % grid].push_back(unit_piece(u));
    for (long long k = 0; k < splits; ++k) {
      Piece a = unit_piece(whole + k), b = a;
      a.t_end = b.t_begin = a.t_begin + (a.t_end - a.t_begin + 1) / 2;
      a.part = 1;
      b.part = 2;
      a.split = b.split = (int32_t)k;
      per_cta[k].push_back(a);
      per_cta[splits + k].push_back(b);
    }
  } else {
    // head dimension 128: whole rounds but the last stay round robin
    const long long lead = head_dim >= 128 ? (units / grid - 1) * grid : 0;
    for (long long u = 0; u < lead; ++u) per_cta[u % grid].push_back(unit_piece(u));
    // the other units' chains cut where the KV tile changes, in head-major chain order
    std::vector<Piece> runs;
    for (long long u = lead; u < units; ++u) {
      const int h = (int)(u / sc.num_slots), slot = (int)(u % sc.num_slots);
      int b = sc.slot_off[slot];
      for (int t = b + 1; t <= sc.slot_off[slot + 1]; ++t)
        if (t == sc.slot_off[slot + 1] || (sc.tasks[t] >> 16) != (sc.tasks[b] >> 16)) {
          runs.push_back({h, b, t});
          b = t;
        }
    }
    // longest first (stable: equal lengths keep the head-major order), each to the CTA
    // with the least work so far (the round-robin rounds gave every CTA the same), the
    // lower index on a tie
    std::stable_sort(runs.begin(), runs.end(), [](const Piece& a, const Piece& b) {
      return a.t_end - a.t_begin > b.t_end - b.t_begin;
    });
    using Load = std::pair<long long, int>;   // (tasks dealt, CTA)
    std::priority_queue<Load, std::vector<Load>, std::greater<Load>> least;
    for (int c = 0; c < grid; ++c) least.push({0, c});
    for (const Piece& pc : runs) {
      Load l = least.top();
      least.pop();
      per_cta[l.second].push_back(pc);
      least.push({l.first + (pc.t_end - pc.t_begin), l.second});
    }
  }
  for (int c = 0; c < grid; ++c) {
    out->cta_off[c + 1] = out->cta_off[c] + (int32_t)per_cta[c].size();
    out->pieces.insert(out->pieces.end(), per_cta[c].begin(), per_cta[c].end());
  }
}

void dealt_orders(const Schedule& sc, int heads, int grid, int head_dim,
                  std::vector<int32_t>* out) {
  const int n = sc.n;
  out->assign((size_t)heads * n * n, -1);
  if (!arrival_ordered(sc)) {
    for (int h = 0; h < heads; ++h)
      std::copy(sc.ord.begin(), sc.ord.end(), out->begin() + (size_t)h * n * n);
    return;
  }
  // (place in the CTA's task sequence, kv) of every partial, per (head, dQ block)
  Dealing dl;
  deal(sc, heads, grid, head_dim, &dl);
  std::vector<std::vector<std::pair<long long, int>>> arrivals((size_t)heads * n);
  for (int cta = 0; cta < grid; ++cta) {
    long long place = 0;
    for (int k = dl.cta_off[cta]; k < dl.cta_off[cta + 1]; ++k) {
      const Piece& pc = dl.pieces[k];
      for (int t = pc.t_begin; t < pc.t_end; ++t, ++place) {
        const int32_t tk = sc.tasks[t];
        arrivals[(size_t)pc.head * n + (tk & 0xffff)].push_back({place, tk >> 16});
      }
    }
  }
  for (size_t hj = 0; hj < arrivals.size(); ++hj) {
    auto& a = arrivals[hj];
    std::sort(a.begin(), a.end());
    const size_t head = hj / n, j = hj % n;
    for (size_t k = 0; k < a.size(); ++k)
      (*out)[(head * n + (size_t)a[k].second) * n + j] = (int32_t)k;
  }
}

bool simulate(const Schedule& sc, int heads, int num_sms, int head_dim, double c, double r,
              double* makespan, std::vector<double>* sm_end) {
  return simulate_ex(sc, heads, num_sms, head_dim, c, r, 0.0, false, makespan, sm_end);
}

bool simulate_ex(const Schedule& sc, int heads, int num_sms, int head_dim, double c, double r,
                 double h, bool overlapped, double* makespan, std::vector<double>* sm_end) {
  const int n = sc.n;
  std::vector<int32_t> ord;
  dealt_orders(sc, heads, num_sms, head_dim, &ord);
  Dealing dl;
  deal(sc, heads, num_sms, head_dim, &dl);
  // who reduces at position k of head h's dQ_j: inv[(h * n + j) * n + k] = kv tile
  std::vector<int32_t> inv((size_t)heads * n * n, -1);
  for (int hd = 0; hd < heads; ++hd)
    for (int i = 0; i < n; ++i)
      for (int j = 0; j < n; ++j) {
        const int o = ord[((size_t)hd * n + i) * n + j];
        if (o >= 0) inv[((size_t)hd * n + j) * n + o] = i;
      }

  // per SM: progress = (piece index into dl.pieces, task index into sc.tasks)
  std::vector<int> piece_pos(num_sms), task_pos(num_sms);
  for (int sm = 0; sm < num_sms; ++sm) {
    piece_pos[sm] = dl.cta_off[sm];
    task_pos[sm] = piece_pos[sm] < dl.cta_off[sm + 1] ? dl.pieces[piece_pos[sm]].t_begin : 0;
  }
  // per SM: end of its last C phase, of its last R phase and of the R phase before that
  std::vector<double> c_last(num_sms, 0.0), r_last(num_sms, 0.0), r_prev(num_sms, 0.0);
  // reduce-end time and SM of (head, kv, q); sentinel -1 = not yet done
  std::vector<double> rend((size_t)heads * n * n, -1.0);
  std::vector<int> rsm((size_t)heads * n * n, -1);

  long long remaining = (long long)heads * (long long)sc.tasks.size();
  while (remaining > 0) {
    bool progress = false;
    for (int sm = 0; sm < num_sms; ++sm) {
      while (piece_pos[sm] < dl.cta_off[sm + 1]) {
        const Piece& pc = dl.pieces[piece_pos[sm]];
        const int head = pc.head;
        const int32_t tk = sc.tasks[task_pos[sm]];
        const int i = tk >> 16, j = tk & 0xffff;
        const int o = ord[((size_t)head * n + i) * n + j];
        double pred_ready = 0.0;
        if (o > 0) {
          const int ip = inv[((size_t)head * n + j) * n + o - 1];
          const size_t pk = ((size_t)head * n + ip) * n + j;
          if (rend[pk] < 0) break;                              // predecessor not done
          pred_ready = rend[pk] + (rsm[pk] == sm ? 0.0 : h);
        }
        // the second half of a split tile ends after its first half (which ends at the
        // task before it in the chain): it adds the first half's dK/dV partial
        double half_ready = 0.0;
        if (pc.part == 2 && task_pos[sm] == pc.t_end - 1) {
          const int32_t ta = sc.tasks[pc.t_begin - 1];
          const size_t ak = ((size_t)head * n + (ta >> 16)) * n + (ta & 0xffff);
          if (rend[ak] < 0) break;
          half_ready = rend[ak];
        }
        double c_end, r_end;
        if (overlapped) {
          c_end = std::max(c_last[sm], r_prev[sm]) + c;
          r_end = std::max(std::max(c_end, r_last[sm]), pred_ready) + r;
        } else {
          c_end = r_last[sm] + c;
          r_end = std::max(c_end, pred_ready) + r;
        }
        r_end = std::max(r_end, half_ready);
        const size_t k = ((size_t)head * n + i) * n + j;
        rend[k] = r_end;
        rsm[k] = sm;
        c_last[sm] = c_end;
        r_prev[sm] = r_last[sm];
        r_last[sm] = r_end;
        --remaining;
        progress = true;
        if (++task_pos[sm] == pc.t_end && ++piece_pos[sm] < dl.cta_off[sm + 1])
          task_pos[sm] = dl.pieces[piece_pos[sm]].t_begin;
      }
    }
    if (!progress) return false;
  }
  double mk = 0.0;
  for (double t : r_last) mk = std::max(mk, t);
  if (makespan) *makespan = mk;
  if (sm_end) *sm_end = r_last;
  return true;
}

}  // namespace dash
