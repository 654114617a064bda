// Host-side DASH schedule tables and the compute/reduce DAG simulator.
//
// Model: "DASH: Deterministic Attention Scheduling for High-throughput Reproducible LLM
// Training", Pith review, sections "Core claim" and "What carries the argument"; task
// orders from the abstract and the Figure 3, 4, 6 and 7 captions.
#pragma once

#include <cstdint>
#include <vector>

namespace dash {

enum { MASK_FULL = 0, MASK_CAUSAL = 1 };
enum { SCHED_ASCENDING = 0, SCHED_DESCENDING = 1, SCHED_SHIFT = 2, SCHED_SYMMETRIC_SHIFT = 3 };

struct Schedule {
  int mask = 0, sched = 0, n = 0;
  int num_slots = 0;                 // chains per head
  int max_chain = 0;                 // longest chain
  std::vector<int32_t> slot_off;     // num_slots + 1
  std::vector<int32_t> tasks;        // (kv << 16) | q, execution order per chain
  std::vector<int32_t> ord;          // n * n; position of KV_i in the dQ_j order, -1 if masked
  std::vector<int32_t> cnt;          // n; contributors per dQ block
};

// Returns 0 and fills `out`, or a positive dash_status_t code.
int build_schedule(int mask, int sched, int n, Schedule* out);

// True when the schedule orders dQ by arrival (its order depends on the dealing).
inline bool arrival_ordered(const Schedule& sc) {
  return sc.sched == SCHED_SHIFT || sc.sched == SCHED_SYMMETRIC_SHIFT;
}

// A run of one head's chain: tasks[t_begin, t_end) of the schedule, for head `head`.
// part 0 covers whole KV tiles; part 1 and 2 are the first and second half of one KV
// tile split over two CTAs (split tile `split`): the first half hands its fp32 dK/dV
// partial to the second, which adds its own and writes dK/dV.
struct Piece {
  int32_t head, t_begin, t_end;
  int32_t part = 0, split = 0;
};

// Most KV tiles one grid splits (bounds the workspace of the split partials).
constexpr int kMaxSplitTiles = 256;

// How many KV tiles deal() splits over two CTAs for `units` units of schedule `sched` (n
// KV tiles per head) on `grid` CTAs: shift's last partial round, r = units mod grid
// units, when 2 r <= grid (and r <= kMaxSplitTiles); otherwise none.
inline long long split_tiles(int sched, int n, long long units, int grid) {
  const long long rem = units % grid;
  if (sched != SCHED_SHIFT || units < grid || rem == 0 || 2 * rem > grid ||
      rem > kMaxSplitTiles || n < 2)
    return 0;
  return rem;
}

// The work of each persistent CTA, in run order: CTA c runs
// pieces[cta_off[c] .. cta_off[c + 1]).
struct Dealing {
  std::vector<int32_t> cta_off;      // grid + 1
  std::vector<Piece> pieces;
};

// How the kernels spread `heads` heads' chains over `grid` persistent CTAs. Round robin
// -- unit u = (head u / num_slots, chain slot u % num_slots) whole to CTA u % grid --
// unless the schedule orders dQ by arrival and the units overrun whole rounds of the grid
// (units % grid != 0 and units > grid). Then round robin would leave some CTAs a whole
// unit more work than the rest, and the chains are instead cut where the KV tile changes
// and the pieces dealt longest first (equal lengths in head-major chain order), each to
// the CTA with the least work dealt so far (the lower index on a tie); a CTA runs its
// pieces in the order dealt. Every KV tile still runs whole on one CTA, in chain order.
// At head dimension 128 the first q - 1 of the q whole rounds stay round robin (whole
// units, head-major) and only the units after them are cut and dealt longest first: a
// round-robin round keeps each head's chains on concurrent CTAs, so its Q/dO tiles and
// dQ accumulator blocks stay in L2, which the twice larger tiles need (at head dimension
// 64 dealing every unit's pieces longest first measured faster).
// Pieces of equal length (shift) are dealt exactly as round robin deals them; there,
// when the last partial round has r units and 2 r <= grid (r <= kMaxSplitTiles), each of
// those r KV tiles is instead split in two halves (the first ceil(len / 2) tasks, then
// the rest): split k's first half runs on CTA k and its second half on CTA r + k, after
// their whole units, so the busiest CTA runs half a unit less and no first half ever
// waits behind a second half.
void deal(const Schedule& sc, int heads, int grid, int head_dim, Dealing* out);

// The dQ order the kernels follow at head dimension `head_dim` when `heads` heads' chains
// are dealt onto `grid` persistent CTAs (deal above): out[(h * n + i) * n + j] = position
// of KV_i's partial in head h's dQ_j order (-1 where the mask removes the task).
//   ascending, descending  -- ascending KV index in every head (`ord` repeated);
//   shift, symmetric shift -- order of arrival: a partial's place in its CTA's task
//                             sequence (the tasks of the CTA's earlier pieces, then its
//                             step), the lower KV index first on a tie.
// When every chain of a head starts together (the pages' setting: one head on n SMs,
// or whole heads per round of the grid) the arrival order is the step order of `ord`.
// When the dealing splits a head over two rounds of the grid, the partials of the chains
// that run in the earlier round come first, so no partial waits for a chain that has not
// started. An arrival-ordered wait always points to a strictly earlier (place, KV index)
// and each CTA runs its tasks in increasing place, so these orders cannot deadlock.
void dealt_orders(const Schedule& sc, int heads, int grid, int head_dim,
                  std::vector<int32_t>* out);

// Event-driven critical path of `heads` heads dealt onto `num_sms` SMs as the kernels
// deal them at head dimension `head_dim` (deal above), with the dQ orders of
// dealt_orders(sc, heads, num_sms, head_dim) -- the orders the kernels follow on a grid of
// num_sms CTAs. Returns false on a cycle (deadlock). sm_end may be null.
bool simulate(const Schedule& sc, int heads, int num_sms, int head_dim, double c, double r,
              double* makespan, std::vector<double>* sm_end);

// The same with synchronisation cost and the two-engine SM (the Pith review's "Where Pith
// is reading between the lines" proposes nonzero edge costs):
//   h          -- cost of handing a dQ block's turn to another SM (0 within one SM);
//   overlapped -- each SM runs C phases in order on one engine and R phases in order on
//                 another, and C of its k-th task waits for R of its (k-2)-th (the
//                 accumulator reuse of a kernel that reads one partial out while the
//                 next is computed); false = C then R, task after task.
// h = 0, overlapped = false is simulate() above.
bool simulate_ex(const Schedule& sc, int heads, int num_sms, int head_dim, double c, double r,
                 double h, bool overlapped, double* makespan, std::vector<double>* sm_end);

}  // namespace dash
