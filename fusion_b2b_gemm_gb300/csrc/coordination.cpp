// Coordination matrix of a register rearrangement (host code).
//
// Patent "数据处理方法、装置、设备及介质" (Alibaba, 2023), Detailed description
// para. 79-91 and Fig. 4: in one exchange round every thread hands out one of
// its values and takes one value, so two threads must never ask the same
// thread in the same round.  The coordination matrix H (n threads x m
// rounds) holds triples (p, q, r): in round j thread i takes value q of
// thread p and keeps it as its value r; within a column the p's differ.
//
// Scheduling: receivers are taken in order; receiver i fills rounds
// 0..m-1 one after another, each time with its first remaining source
// (in the order of its own values) whose thread is still free in that round.
// This greedy order reproduces the patent's first row for the tf32 example.
// When it gets stuck, the matrix is rebuilt round by round from perfect
// matchings of the receiver/sender multigraph, which always exist because
// every thread sends and receives exactly m values (a regular bipartite
// multigraph splits into m perfect matchings).
#include <cstdint>
#include <vector>

#include "b2b.h"

namespace {

struct Edge {
  int p, q, r;  // sender, sender's value, receiver's slot
};

bool greedy(int n, int m, const std::vector<std::vector<Edge>>& need, int* P, int* Q, int* R) {
  std::vector<std::vector<char>> busy(m, std::vector<char>(n, 0));  // busy[j][p]
  for (int i = 0; i < n; ++i) {
    std::vector<char> done(m, 0);
    for (int j = 0; j < m; ++j) {
      int pick = -1;
      for (int k = 0; k < m; ++k)
        if (!done[k] && !busy[j][need[i][k].p]) {
          pick = k;
          break;
        }
      if (pick < 0) return false;
      done[pick] = 1;
      busy[j][need[i][pick].p] = 1;
      P[i * m + j] = need[i][pick].p;
      Q[i * m + j] = need[i][pick].q;
      R[i * m + j] = need[i][pick].r;
    }
  }
  return true;
}

// Kuhn's augmenting path on the remaining edges (receiver -> sender).
bool augment(int i, const std::vector<std::vector<Edge>>& need, const std::vector<std::vector<char>>& used,
             std::vector<char>& seen, std::vector<int>& owner, std::vector<int>& via) {
  const int m = static_cast<int>(need[i].size());
  for (int k = 0; k < m; ++k) {
    if (used[i][k]) continue;
    const int p = need[i][k].p;
    if (seen[p]) continue;
    seen[p] = 1;
    if (owner[p] < 0 || augment(owner[p], need, used, seen, owner, via)) {
      owner[p] = i;
      via[p] = k;
      return true;
    }
  }
  return false;
}

bool by_matchings(int n, int m, const std::vector<std::vector<Edge>>& need, int* P, int* Q, int* R) {
  std::vector<std::vector<char>> used(n, std::vector<char>(m, 0));
  for (int j = 0; j < m; ++j) {
    std::vector<int> owner(n, -1), via(n, -1);
    for (int i = 0; i < n; ++i) {
      std::vector<char> seen(n, 0);
      if (!augment(i, need, used, seen, owner, via)) return false;
    }
    for (int p = 0; p < n; ++p) {
      const int i = owner[p], k = via[p];
      used[i][k] = 1;
      P[i * m + j] = need[i][k].p;
      Q[i * m + j] = need[i][k].q;
      R[i * m + j] = need[i][k].r;
    }
  }
  return true;
}

}  // namespace

extern "C" b2b_status_t b2b_coordination_matrix(int n, int m, const int* src_thread,
                                                const int* src_reg, int* P, int* Q, int* R) {
  if (n < 1 || m < 1 || n > 1024 || m > 1024) return B2B_ERR_INVALID_ARG;
  if (!src_thread || !src_reg || !P || !Q || !R) return B2B_ERR_INVALID_ARG;
  std::vector<char> taken(static_cast<size_t>(n) * m, 0);
  std::vector<std::vector<Edge>> need(n, std::vector<Edge>(m));
  for (int i = 0; i < n; ++i)
    for (int r = 0; r < m; ++r) {
      const int p = src_thread[i * m + r], q = src_reg[i * m + r];
      if (p < 0 || p >= n || q < 0 || q >= m) return B2B_ERR_INVALID_ARG;
      char& t = taken[static_cast<size_t>(p) * m + q];
      if (t) return B2B_ERR_INVALID_ARG;  // a source value used twice
      t = 1;
      need[i][r] = Edge{p, q, r};
    }
  // every source is used exactly once, so every thread sends exactly m values
  if (greedy(n, m, need, P, Q, R)) return B2B_OK;
  if (by_matchings(n, m, need, P, Q, R)) return B2B_OK;
  return B2B_ERR_UNSUPPORTED;
}
