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

bool make_pair_split(int heads, int ctas, PairSplit* sp) {
  const int pairs = ctas / 2;
  if (pairs < 1 || ctas > kMaxCtas) return false;
  for (int c = 0; c <= pairs; ++c) sp->head[c] = (uint16_t)((int64_t)heads * c / pairs);
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

// Relative time of a single-head rope box (eight M = 64 MMAs on 16 KiB)
// against a 128-row box (four M = 128 MMAs), as a fraction.
constexpr int kSingleCostNum = 5, kSingleCostDen = 4;

// Fills the split for one rope unit shape; returns the most loaded CTA's
// estimated time in 128-row boxes x kSingleCostDen, or -1 if some pair would
// get more than two heads.
int64_t fill_wide_split(int heads, int pairs, int single, WideSplit* sp) {
  sp->single = single;
  for (int c = 0; c <= pairs; ++c) sp->head[c] = (uint16_t)((int64_t)heads * c / pairs);
  for (int c = 0; c < pairs; ++c)
    if (sp->head[c + 1] - sp->head[c] > 2) return -1;
  // ROPE units (two heads' rope rows, 12 boxes of 16 KiB per CTA, or one
  // head's, 6 boxes) fill every pair up to an even share of the bytes; a
  // head's NOPE + ABS units are 16 boxes per CTA (its nope rows' K half and
  // its half of W_UK^T).
  const int ropes = single ? heads : (heads + 1) / 2;
  const int64_t hb = kWideHeadBoxes, rb = single ? kWideSingleBoxes : kWideRopeBoxes;
  const int64_t total = (int64_t)heads * hb + (int64_t)ropes * rb;
  int64_t head_bytes = 0, most = 0;
  int prev = 0;
  sp->rope[0] = 0;
  for (int c = 0; c < pairs; ++c) {
    const int nh = sp->head[c + 1] - sp->head[c];
    head_bytes += (int64_t)nh * hb;
    int64_t r = (total * (c + 1) / pairs - head_bytes + rb / 2) / rb;
    if (r < prev) r = prev;
    if (r > ropes) r = ropes;
    if (c == pairs - 1) r = ropes;
    sp->rope[c + 1] = (uint16_t)r;
    const int64_t cost = (int64_t)nh * hb * kSingleCostDen +
                         (r - prev) * rb * (single ? kSingleCostNum : kSingleCostDen);
    if (cost > most) most = cost;
    prev = (int)r;
  }
  return most;
}

}  // namespace

bool make_wide_split(int heads, int ctas, WideSplit* sp) {
  const int pairs = ctas / 2;
  sp->single = 0;
  if (pairs < 1 || ctas > kMaxCtas) return false;
  WideSplit one;
  const int64_t two_cost = fill_wide_split(heads, pairs, 0, sp);
  const int64_t one_cost = fill_wide_split(heads, pairs, 1, &one);
  if (two_cost < 0) return false;
  if (one_cost >= 0 && one_cost < two_cost) *sp = one;
  return true;
}

}  // namespace mla
