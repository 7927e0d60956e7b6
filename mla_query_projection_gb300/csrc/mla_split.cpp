// mla_split.cpp - the create-time work splits of the absorbing kernels
// (host code only, no CUDA calls).  Each split hands every CTA (or cluster
// pair) a contiguous run of heads or tasks and of rope rows, sized so the
// bytes each CTA streams are as even as the units allow: the weights of a
// decode step (page "mla.query", class MlaQuery: W_QB rows and W_UK) are
// read once, and the step lasts as long as its most loaded CTA.
#include "mla_internal.h"

namespace mla {

void make_abs_split(int heads, int ctas, AbsSplit* sp) {
  // tasks: even split; rope rows: fill each CTA up to an even share of bytes
  const int64_t tasks = (int64_t)heads * kTasksPerHead, rope = (int64_t)heads * kRope;
  const int64_t tb = kTaskRows * kRowBytes + kTaskUkBytes, rb = kRowBytes;
  const int64_t total = tasks * tb + rope * rb;
  int prev = 0;
  for (int i = 0; i <= ctas; ++i) {
    const int64_t t = tasks * i / ctas;
    sp->task[i] = (uint16_t)t;
    int64_t r = (total * i / ctas - t * tb + rb / 2) / rb;
    if (r < prev) r = prev;
    if (r > rope) r = rope;
    if (i == ctas) r = rope;
    sp->rope[i] = (uint16_t)r;
    prev = (int)r;
  }
}

bool make_pair_split(int heads, int ctas, bool heads_first, PairSplit* sp) {
  const int pairs = ctas / 2;
  if (pairs < 1 || ctas > kMaxCtas) return false;
  for (int c = 0; c <= pairs; ++c)
    sp->head[c] = heads_first && heads <= pairs ? (uint16_t)(c < heads ? c : heads)
                                                : (uint16_t)((int64_t)heads * c / pairs);
  for (int c = 0; c < pairs; ++c)
    if (sp->head[c + 1] - sp->head[c] > 2) return false;
  // rope rows fill every CTA up to an even share of the bytes
  const int64_t tb = (int64_t)4 * (kTaskRows * kRowBytes + kTaskUkBytes);  // one head's tasks
  const int64_t rb = kRowBytes, rope = (int64_t)heads * kRope;
  const int64_t total = (int64_t)heads * 2 * tb + rope * rb;
  int64_t task_bytes = 0;
  int prev = 0;
  sp->rope[0] = 0;
  for (int i = 0; i < ctas; ++i) {
    task_bytes += (int64_t)(sp->head[i / 2 + 1] - sp->head[i / 2]) * tb;
    int64_t r = (total * (i + 1) / ctas - task_bytes + rb / 2) / rb;
    if (r < prev) r = prev;
    if (r > rope) r = rope;
    if (i == ctas - 1) r = rope;
    sp->rope[i + 1] = (uint16_t)r;
    prev = (int)r;
  }
  return true;
}

int64_t pair_split_max_bytes(int ctas, const PairSplit& sp) {
  const int64_t tb = (int64_t)4 * (kTaskRows * kRowBytes + kTaskUkBytes);  // half a head
  int64_t most = 0;
  for (int i = 0; i < ctas; ++i) {
    const int64_t b = (int64_t)(sp.head[i / 2 + 1] - sp.head[i / 2]) * tb +
                      (int64_t)(sp.rope[i + 1] - sp.rope[i]) * kRowBytes;
    if (b > most) most = b;
  }
  return most;
}

bool make_small_split(int heads, int ctas, int cluster, SmallSplit* sp) {
  if (cluster != 2 && cluster != 4 && cluster != 8) return false;
  if (ctas < cluster || ctas % cluster != 0 || ctas > kMaxCtas) return false;
  const int groups = ctas / cluster;
  sp->cluster = cluster;
  for (int g = 0; g <= groups; ++g) sp->head[g] = (uint16_t)((int64_t)heads * g / groups);
  for (int g = 0; g < groups; ++g)
    if (sp->head[g + 1] - sp->head[g] > 2) return false;
  // rope rows fill every CTA up to an even share of the bytes
  const int64_t tb = (int64_t)(kNope / cluster) * (kRowBytes + kKvLora * 2);  // a head's rows
  const int64_t rb = kRowBytes, rope = (int64_t)heads * kRope;
  const int64_t total = (int64_t)heads * cluster * tb + rope * rb;
  int64_t task_bytes = 0;
  int prev = 0;
  sp->rope[0] = 0;
  for (int i = 0; i < ctas; ++i) {
    task_bytes += (int64_t)(sp->head[i / cluster + 1] - sp->head[i / cluster]) * tb;
    int64_t r = (total * (i + 1) / ctas - task_bytes + rb / 2) / rb;
    if (r < prev) r = prev;
    if (r > rope) r = rope;
    if (i == ctas - 1) r = rope;
    sp->rope[i + 1] = (uint16_t)r;
    prev = (int)r;
  }
  return true;
}

int64_t small_split_max_bytes(int heads, int ctas, const SmallSplit& sp) {
  (void)heads;
  const int c = sp.cluster;
  const int64_t tb = (int64_t)(kNope / c) * (kRowBytes + kKvLora * 2);
  int64_t most = 0;
  for (int i = 0; i < ctas; ++i) {
    const int64_t b = (int64_t)(sp.head[i / c + 1] - sp.head[i / c]) * tb +
                      (int64_t)(sp.rope[i + 1] - sp.rope[i]) * kRowBytes;
    if (b > most) most = b;
  }
  return most;
}

int choose_small_split(int heads, int num_sms, const int* max_clusters, SmallSplit* sp) {
  int best_ctas = 0;
  int64_t best = 0;
  SmallSplit trial;
  for (int k = 0, c = 2; c <= 8; ++k, c *= 2) {
    int groups = num_sms / c;
    if (max_clusters != nullptr && max_clusters[k] < 0) continue;  // cannot run
    if (max_clusters != nullptr && max_clusters[k] > 0 && max_clusters[k] < groups)
      groups = max_clusters[k];
    const int ctas = groups * c;
    if (ctas < c || !make_small_split(heads, ctas, c, &trial)) continue;
    const int64_t most = small_split_max_bytes(heads, ctas, trial);
    if (best_ctas == 0 || most < best) {  // ties keep the smaller cluster
      best = most;
      best_ctas = ctas;
      *sp = trial;
    }
  }
  return best_ctas;
}

namespace {

// Estimated time of a CTA's units in quarter boxes: a 128-row box (a head's
// NOPE / ABS box, or a two-head rope box: four M = 128 MMAs on 16 KiB) costs
// 4, a one-head rope box (eight M = 64 MMAs on 16 KiB) 5.
constexpr int64_t kHeadCost = (int64_t)kWideHeadBoxes * 4;   // 64
constexpr int64_t kDoubleCost = (int64_t)kWideRopeBoxes * 4;  // 48
constexpr int64_t kSingleCost = (int64_t)kWideSingleBoxes * 5;  // 30

// Fills the split for `ndouble` two-head rope units (and one-head units for
// the heads past them): each unit, two-head units first, goes to the pair
// with the least estimated time so far (ties: the lower index).  Returns the
// most loaded pair's estimate, or -1 if some pair would get more than two
// heads.
int64_t fill_wide_split(int heads, int pairs, int ndouble, WideSplit* sp) {
  if (pairs > kMaxCtas / 2) return -1;
  for (int c = 0; c <= pairs; ++c) sp->head[c] = (uint16_t)((int64_t)heads * c / pairs);
  int64_t load[kMaxCtas / 2];
  int nd[kMaxCtas / 2], ns[kMaxCtas / 2];
  for (int c = 0; c < pairs; ++c) {
    const int nh = sp->head[c + 1] - sp->head[c];
    if (nh > 2) return -1;
    load[c] = nh * kHeadCost;
    nd[c] = ns[c] = 0;
  }
  const int singles = heads > 2 * ndouble ? heads - 2 * ndouble : 0;
  for (int k = 0; k < ndouble + singles; ++k) {
    int best = 0;
    for (int c = 1; c < pairs; ++c)
      if (load[c] < load[best]) best = c;
    if (k < ndouble) {
      load[best] += kDoubleCost;
      ++nd[best];
    } else {
      load[best] += kSingleCost;
      ++ns[best];
    }
  }
  sp->ndouble = ndouble;
  sp->dbl[0] = sp->sgl[0] = 0;
  int64_t most = 0;
  for (int c = 0; c < pairs; ++c) {
    sp->dbl[c + 1] = (uint16_t)(sp->dbl[c] + nd[c]);
    sp->sgl[c + 1] = (uint16_t)(sp->sgl[c] + ns[c]);
    if (load[c] > most) most = load[c];
  }
  return most;
}

}  // namespace

bool make_wide_split(int heads, int ctas, WideSplit* sp) {
  const int pairs = ctas / 2;
  if (pairs < 1 || ctas > kMaxCtas || heads < 1) return false;
  // the fewest quarter boxes on the most loaded pair over every mix of the
  // two rope-unit shapes; ties keep, in this order, two-head units only,
  // one-head units only (measured: at 64 heads, 14.46 against 14.83 us at
  // B = 64 for a mix of the same estimate), then more two-head units
  const int most_double = (heads + 1) / 2;
  int64_t best = -1;
  WideSplit trial;
  for (int k = 0; k <= most_double; ++k) {
    const int d = k == 0 ? most_double : k == 1 ? 0 : most_double + 1 - k;
    if (k > 0 && d == most_double) continue;
    const int64_t cost = fill_wide_split(heads, pairs, d, &trial);
    if (cost < 0) return false;
    if (best < 0 || cost < best) {
      best = cost;
      *sp = trial;
    }
  }
  return true;
}

}  // namespace mla
