// Verify prices and the StairCut cut -- host code
// [Drafters and tree verify, §StairCut: the node count, calculated each round;
// §StairCut on Flash-Next, and the shared price files].
//
// V(rows) comes from a table of measured verify prices keyed by context class
// and kind (chain or tree): a context takes the nearest lower class (the lowest
// when it is below all of them); rows between two measured counts interpolate;
// rows past the last measured count add step_ms a row, else the slope of the
// last two counts; rows below the first measured count take its price; and a
// price never falls with more rows.  The table follows the live prices: an
// observed count moves toward each observation by an exponential average of
// weight 0.1, and the counts never observed move by the learned offset (the
// same average of observed minus table price).
//
// The cut admits the drafted nodes in the order of the drafter's score, each
// with the ancestors it needs, and tries the counts 7, 15, 23 and 31 nodes and
// the whole candidate, keeping the one that maximises
//     (1 + min(sum q, n)) / (V(n + 1 rows) + draft + commit)
// (a chain pays the rollback weighted by 1 - q of its deepest kept node
// instead of the commit; equal values keep the smaller count).
//
// Built with floating-point contraction off, so that every price is the same
// double on every host.
#include <cmath>
#include <cstdint>

#include "../../include/tv.h"

namespace {

constexpr double kEma = 0.1;
constexpr int kCuts[4] = {7, 15, 23, 31};

bool valid_table(const tv_price_table* t) {
  if (!t || t->n_classes < 1 || t->n_classes > TV_PRICE_MAX_CLASSES) return false;
  for (int c = 1; c < t->n_classes; ++c)
    if (t->class_ctx[c] <= t->class_ctx[c - 1]) return false;
  return std::isfinite(t->step_ms) && t->step_ms >= 0.0;
}

int class_of(const tv_price_table* t, int32_t context) {
  int c = 0;
  for (int i = 0; i < t->n_classes; ++i)
    if (t->class_ctx[i] <= context) c = i;
  return c;
}

// the table's price of one count, before the online state and the never-falls rule
double raw_price(const tv_price_table* t, int c, int kind, int rows) {
  const double* p = t->prior[c][kind];
  int xs[TV_PRICE_MAX_ROWS + 1];
  int np = 0;
  for (int r = 1; r <= TV_PRICE_MAX_ROWS; ++r)
    if (!std::isnan(p[r])) xs[np++] = r;
  if (np == 0) return 0.0;
  if (rows <= xs[0]) return p[xs[0]];
  for (int i = 0; i + 1 < np; ++i) {
    const int x0 = xs[i], x1 = xs[i + 1];
    if (x0 <= rows && rows <= x1) {
      const double y0 = p[x0], y1 = p[x1];
      return y0 + (y1 - y0) * (double)(rows - x0) / (double)(x1 - x0);
    }
  }
  const int xl = xs[np - 1];
  if (t->step_ms > 0.0 || np == 1) return p[xl] + t->step_ms * (double)(rows - xl);
  const int xp = xs[np - 2];
  const double slope = (p[xl] - p[xp]) / (double)(xl - xp);
  return p[xl] + slope * (double)(rows - xl);
}

double current_price(const tv_price_table* t, int c, int kind, int rows) {
  const double live = t->live[c][kind][rows];
  if (!std::isnan(live)) return live;
  return raw_price(t, c, kind, rows) + t->offset[c][kind];
}

double price(const tv_price_table* t, int32_t context, int kind, int rows) {
  const int c = class_of(t, context);
  double m = current_price(t, c, kind, 1);
  for (int r = 2; r <= rows; ++r) {
    const double v = current_price(t, c, kind, r);
    if (v > m) m = v;
  }
  return m;
}

}  // namespace

extern "C" {

int tv_price_init(tv_price_table* t) {
  if (!t) return TV_E_ARG;
  t->n_classes = 0;
  t->step_ms = 0.0;
  for (int c = 0; c < TV_PRICE_MAX_CLASSES; ++c) {
    t->class_ctx[c] = 0;
    for (int k = 0; k < 2; ++k) {
      t->offset[c][k] = 0.0;
      for (int r = 0; r <= TV_PRICE_MAX_ROWS; ++r) {
        t->prior[c][k][r] = NAN;
        t->live[c][k][r] = NAN;
      }
    }
  }
  return TV_OK;
}

int tv_price_lookup(const tv_price_table* t, int32_t context, int32_t kind, int32_t rows, double* ms) {
  if (!valid_table(t) || !ms || (kind != TV_KIND_CHAIN && kind != TV_KIND_TREE)) return TV_E_ARG;
  if (rows < 1 || rows > TV_PRICE_MAX_ROWS) return TV_E_ROWS;
  *ms = price(t, context, kind, rows);
  return TV_OK;
}

int tv_price_observe(tv_price_table* t, int32_t context, int32_t kind, int32_t rows, double ms) {
  if (!valid_table(t) || (kind != TV_KIND_CHAIN && kind != TV_KIND_TREE) || !std::isfinite(ms)) return TV_E_ARG;
  if (rows < 1 || rows > TV_PRICE_MAX_ROWS) return TV_E_ROWS;
  const int c = class_of(t, context);
  const double prior = raw_price(t, c, kind, rows);
  const double old = current_price(t, c, kind, rows);
  t->live[c][kind][rows] = old + kEma * (ms - old);
  const double off = t->offset[c][kind];
  t->offset[c][kind] = off + kEma * ((ms - prior) - off);
  return TV_OK;
}

int tv_staircut(const int32_t* parent, const float* q, const float* score, int32_t n, int32_t kind,
                const tv_price_table* t, int32_t context, double draft_ms, double commit_ms, double rollback_ms,
                int32_t* keep, int32_t* n_keep, double* value) {
  if (!parent || !q || !score || !keep || !n_keep || !value || !valid_table(t) ||
      (kind != TV_KIND_CHAIN && kind != TV_KIND_TREE))
    return TV_E_ARG;
  if (n < 1 || n > TV_PRICE_MAX_ROWS) return TV_E_ROWS;
  if (parent[0] != -1) return TV_E_ORDER;
  for (int i = 1; i < n; ++i)
    if (parent[i] < 0 || parent[i] >= i) return TV_E_ORDER;
  // nodes by score, highest first (lower index on ties): insertion sort of <= 31
  int by_score[TV_PRICE_MAX_ROWS];
  int m = 0;
  for (int i = 1; i < n; ++i) {
    int j = m++;
    while (j > 0 && (score[by_score[j - 1]] < score[i] ||
                     (score[by_score[j - 1]] == score[i] && by_score[j - 1] > i))) {
      by_score[j] = by_score[j - 1];
      --j;
    }
    by_score[j] = i;
  }
  // admission order: each node preceded by its ancestors not yet admitted
  int order[TV_PRICE_MAX_ROWS];
  bool seen[TV_PRICE_MAX_ROWS] = {true};
  int total = 0;
  for (int k = 0; k < m; ++k) {
    int chain[TV_PRICE_MAX_ROWS];
    int len = 0;
    for (int a = by_score[k]; !seen[a]; a = parent[a]) chain[len++] = a;
    for (int i = len - 1; i >= 0; --i) {
      seen[chain[i]] = true;
      order[total++] = chain[i];
    }
  }
  // candidate counts, ascending: 7, 15, 23, 31 up to the candidate, then the whole
  int counts[5];
  int nc = 0;
  const int whole = total < kCuts[3] ? total : kCuts[3];
  for (int c : kCuts)
    if (c <= total && c != whole) counts[nc++] = c;
  counts[nc++] = whole;
  for (int i = nc - 1; i > 0 && counts[i] < counts[i - 1]; --i) {   // whole may sit below a cut
    const int tmp = counts[i];
    counts[i] = counts[i - 1];
    counts[i - 1] = tmp;
  }
  double best = -INFINITY;
  int best_cnt = 0;
  for (int i = 0; i < nc; ++i) {
    const int cnt = counts[i];
    double sq = 0.0;
    for (int k = 0; k < cnt; ++k) sq += (double)(q[order[k]] < 1.f ? q[order[k]] : 1.f);
    const double gain = 1.0 + (sq < (double)cnt ? sq : (double)cnt);
    double cost = price(t, context, kind, cnt + 1) + draft_ms;
    if (kind == TV_KIND_CHAIN) {
      const double ql = cnt > 0 ? (double)(q[order[cnt - 1]] < 1.f ? q[order[cnt - 1]] : 1.f) : 1.0;
      cost += (1.0 - ql) * rollback_ms;
    } else {
      cost += commit_ms;
    }
    const double v = gain / cost;
    if (v > best) {
      best = v;
      best_cnt = cnt;
    }
  }
  for (int k = 0; k < best_cnt; ++k) keep[k] = order[k];
  *n_keep = best_cnt;
  *value = best;
  return TV_OK;
}

}  // extern "C"
