// Host builders of the packed candidate tree.
//   medusa_tree_cartesian: the Cartesian product of the per-head top-s_k ("Medusa: Simple
//     LLM Inference Acceleration Framework with Multiple Decoding Heads" §3.4 Tree
//     Attention, Step 2).
//   medusa_tree_greedy: the optimized sparse tree (same page, §3.4 "Optimized Tree
//     Construction"; "Accelerating LLM Inference with Speculative Decoding: Notes on
//     Medusa", section 4): E[L] is the sum over all tree nodes of the product of the
//     marginal accuracies on the node's path, and nodes are added one at a time, always
//     the frontier node with the largest path product (ties to the smaller rank path).
// Both return the canonical packing: root first, then nodes by depth, then by rank path,
// so every parent precedes its children.
#include <algorithm>
#include <vector>

#include "../../include/medusa.h"

namespace {

typedef std::vector<int> Path;

bool path_less(const Path& x, const Path& y) {        // depth first, then lexicographic
  if (x.size() != y.size()) return x.size() < y.size();
  return x < y;
}

int pack(std::vector<Path> paths, int max_nodes, int32_t* parent, int32_t* rank) {
  std::sort(paths.begin(), paths.end(), path_less);
  paths.erase(std::unique(paths.begin(), paths.end()), paths.end());
  const int n1 = (int)paths.size() + 1;
  if (n1 > max_nodes) return MEDUSA_ERR_INVALID;
  parent[0] = -1;
  rank[0] = 0;
  for (int n = 1; n < n1; ++n) {
    const Path& p = paths[n - 1];
    rank[n] = p.back();
    if (p.size() == 1) {
      parent[n] = 0;
      continue;
    }
    const Path up(p.begin(), p.end() - 1);
    // the parent is an earlier packed node: binary search in the sorted list
    auto it = std::lower_bound(paths.begin(), paths.begin() + (n - 1), up, path_less);
    if (it == paths.begin() + (n - 1) || *it != up) return MEDUSA_ERR_INVALID;
    parent[n] = (int32_t)(it - paths.begin()) + 1;
  }
  return n1;
}

}  // namespace

extern "C" int medusa_tree_cartesian(int K, const int* s, int max_nodes, int32_t* parent,
                                     int32_t* rank) {
  if (K < 1 || K > MEDUSA_MAX_HEADS || !s || !parent || !rank) return MEDUSA_ERR_INVALID;
  for (int k = 0; k < K; ++k)
    if (s[k] < 1 || s[k] > MEDUSA_MAX_TOPS) return MEDUSA_ERR_INVALID;
  std::vector<Path> all, level(1);
  for (int k = 0; k < K; ++k) {
    std::vector<Path> next;
    for (const Path& p : level)
      for (int i = 0; i < s[k]; ++i) {
        Path c = p;
        c.push_back(i);
        next.push_back(c);
        if ((long)all.size() + (long)next.size() + 1 > (long)max_nodes) return MEDUSA_ERR_INVALID;
      }
    all.insert(all.end(), next.begin(), next.end());
    level.swap(next);
  }
  return pack(all, max_nodes, parent, rank);
}

extern "C" int medusa_tree_greedy(int K, const int* s, int smax, const double* a, int N,
                                  int32_t* parent, int32_t* rank) {
  if (K < 1 || K > MEDUSA_MAX_HEADS || !s || !a || !parent || !rank || N < 0)
    return MEDUSA_ERR_INVALID;
  for (int k = 0; k < K; ++k)
    if (s[k] < 1 || s[k] > smax) return MEDUSA_ERR_INVALID;
  struct Cand { Path p; double score; };
  std::vector<Cand> frontier;
  for (int i = 0; i < s[0]; ++i) frontier.push_back({Path{i}, a[i]});
  std::vector<Path> chosen;
  while ((int)chosen.size() < N && !frontier.empty()) {
    size_t best = 0;
    for (size_t c = 1; c < frontier.size(); ++c) {
      const Cand& x = frontier[c];
      const Cand& y = frontier[best];
      if (x.score > y.score || (x.score == y.score && x.p < y.p)) best = c;
    }
    Cand pick = frontier[best];
    frontier.erase(frontier.begin() + best);
    chosen.push_back(pick.p);
    const int depth = (int)pick.p.size();
    if (depth < K)
      for (int i = 0; i < s[depth]; ++i) {
        Path c = pick.p;
        c.push_back(i);
        frontier.push_back({c, pick.score * a[depth * smax + i]});
      }
  }
  return pack(chosen, N + 1, parent, rank);
}

extern "C" int medusa_tree_size_choose(const double* expected, int max_n, const int* sizes,
                                       const double* step_ms, int n) {
  if (!expected || !sizes || !step_ms || n < 1 || max_n < 0) return MEDUSA_ERR_INVALID;
  int best = -1;
  double best_rate = 0.0;
  for (int i = 0; i < n; ++i) {
    if (sizes[i] < 0 || sizes[i] > max_n || !(step_ms[i] > 0.0)) return MEDUSA_ERR_INVALID;
    const double rate = (1.0 + expected[sizes[i]]) / step_ms[i];     // tokens per ms
    if (best < 0 || rate > best_rate || (rate == best_rate && sizes[i] < sizes[best])) {
      best = i;
      best_rate = rate;
    }
  }
  return best;
}
