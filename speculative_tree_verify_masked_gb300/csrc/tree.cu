// Draft-tree preparation, the accept walk and length bookkeeping.
//
// Tree preparation derives, per node, the depth, the ancestor-or-self bitmask
// (the tree mask of the merged draft tree, "One request, end to end" 2.6),
// the ancestor at every depth (the rows a node attends to past the context)
// and the traversal order of the recurrent layers.
//
// Recurrent traversal.  Every node's Gated DeltaNet state is its parent's
// state advanced by one token, so a depth-first walk needs the parent's state
// only until its last child starts.  The walk visits the children of a node
// with several children lightest subtree first and the heaviest last; the
// parent's state is saved in a slot while the light subtrees run and the
// heaviest child continues from that slot with the slot released.  Each saved
// slot therefore sits above a light subtree of at most half the enclosing
// size, so a tree of n nodes needs at most floor(log2(n / 3)) + 1 slots:
// 5 for 64 nodes.  The order never changes any node's arithmetic: each state
// is always exactly one step from its parent's.
#include "common.cuh"
#include "host.hpp"

namespace tv {

__global__ void tree_prepare_kernel(const int32_t* __restrict__ node_off, const int32_t* __restrict__ parent,
                                    void* meta, int32_t* status, int n_seq, int n_total, int n_max) {
  const int s = threadIdx.x;
  if (s >= n_seq) return;
  MetaView mv = meta_view(meta, n_total);
  const int off = node_off[s];
  const int end = node_off[s + 1];
  const int n = end - off;
  bool ok = off >= 0 && end <= n_total && n >= 1 && n <= n_max && n <= TV_MAX_NODES &&
            (s > 0 || off == 0) && (s < n_seq - 1 || end == n_total);
  int par[TV_MAX_NODES], dep[TV_MAX_NODES], nch[TV_MAX_NODES], size[TV_MAX_NODES], heavy[TV_MAX_NODES];
  uint64_t anc[TV_MAX_NODES];
  int max_depth = 0;
  if (ok) {
    for (int i = 0; i < n && ok; i++) {
      const int p = parent[off + i];
      if (i == 0) {
        ok = (p == -1);
        par[0] = -1;
        dep[0] = 0;
        anc[0] = 1ull;
      } else {
        ok = (p >= 0 && p < i);
        if (ok) {
          par[i] = p;
          dep[i] = dep[p] + 1;
          anc[i] = anc[p] | (1ull << i);
          ok = dep[i] < TV_MAX_PATH;
          max_depth = dep[i] > max_depth ? dep[i] : max_depth;
        }
      }
    }
  }
  if (!ok) {
    set_status(status, TV_ERR_TREE);
    mv.seq[s] = SeqInfo{0, off, 0, 0};
    return;
  }
  for (int i = 0; i < n; i++) {
    mv.anc[off + i] = anc[i];
    mv.depth[off + i] = dep[i];
    int8_t* row = mv.anc_at + static_cast<size_t>(off + i) * TV_MAX_PATH;
    for (int e = 0; e < TV_MAX_PATH; e++) row[e] = -1;
    for (int j = i; j != -1; j = par[j]) row[dep[j]] = static_cast<int8_t>(j);
  }
  // subtree sizes and heaviest child (lowest index among equals)
  for (int i = 0; i < n; i++) {
    nch[i] = 0;
    size[i] = 1;
    heavy[i] = -1;
  }
  for (int i = n - 1; i >= 1; i--) size[par[i]] += size[i];
  for (int i = 1; i < n; i++) {
    const int p = par[i];
    nch[p]++;
    if (heavy[p] < 0 || size[i] > size[heavy[p]]) heavy[p] = i;
  }
  // depth-first walk, lightest subtrees first; stack entries (node, src, level)
  int st_node[TV_MAX_NODES], st_src[TV_MAX_NODES], st_lvl[TV_MAX_NODES];
  int sp = 0, k = 0, max_slot = -1;
  st_node[0] = 0;
  st_src[0] = 0;
  st_lvl[0] = 0;
  sp = 1;
  while (sp > 0 && ok) {
    sp--;
    const int u = st_node[sp], src = st_src[sp], lv = st_lvl[sp];
    int save = 0;
    if (nch[u] >= 2) {
      if (lv >= kMaxSlots) {
        ok = false;
        break;
      }
      save = 1 + lv;
      max_slot = lv > max_slot ? lv : max_slot;
    }
    mv.sched[off + k] = sched_encode(u, src, save, nch[u] > 0 ? 1 : 0);
    k++;
    if (nch[u] == 0) continue;
    if (nch[u] == 1) {
      st_node[sp] = heavy[u];
      st_src[sp] = 0;
      st_lvl[sp] = lv;
      sp++;
      continue;
    }
    st_node[sp] = heavy[u];
    st_src[sp] = 1 + lv;
    st_lvl[sp] = lv;
    sp++;
    int first_light = -1;
    for (int c = n - 1; c >= 1; c--)
      if (par[c] == u && c != heavy[u]) first_light = c;
    for (int c = n - 1; c >= 1; c--) {
      if (par[c] == u && c != heavy[u]) {
        st_node[sp] = c;
        st_src[sp] = (c == first_light) ? 0 : 1 + lv;
        st_lvl[sp] = lv + 1;
        sp++;
      }
    }
  }
  if (!ok || k != n) {
    set_status(status, TV_ERR_TREE);
    mv.seq[s] = SeqInfo{0, off, 0, 0};
    return;
  }
  mv.seq[s] = SeqInfo{n, off, max_depth, max_slot + 1};
}

// Longest agreeing path plus one token ("One request, end to end" 2.6).
__global__ void accept_kernel(const int32_t* __restrict__ tok, const int32_t* __restrict__ greedy,
                              const void* meta, int n_seq, int n_total, int32_t* path, int32_t* acc_len,
                              int32_t* bonus, int32_t* status) {
  const int s = threadIdx.x;
  if (s >= n_seq) return;
  int32_t* prow = path + s * TV_MAX_PATH;
  if (status_bad(status)) {
    for (int e = 0; e < TV_MAX_PATH; e++) prow[e] = -1;
    acc_len[s] = 0;
    bonus[s] = -1;
    return;
  }
  MetaView mv = meta_view(const_cast<void*>(meta), n_total);
  const SeqInfo info = mv.seq[s];
  const int n = info.n, off = info.off;
  bool agree[TV_MAX_NODES];
  agree[0] = true;
  int best = 0, best_depth = 0;
  for (int i = 1; i < n; i++) {
    const int d = mv.depth[off + i];
    const int p = mv.anc_at[static_cast<size_t>(off + i) * TV_MAX_PATH + d - 1];
    agree[i] = agree[p] && tok[off + i] == greedy[off + p];
    if (agree[i] && d > best_depth) {
      best = i;
      best_depth = d;
    }
  }
  const int a = best_depth + 1;
  const int8_t* arow = mv.anc_at + static_cast<size_t>(off + best) * TV_MAX_PATH;
  for (int e = 0; e < TV_MAX_PATH; e++) prow[e] = e < a ? arow[e] : -1;
  acc_len[s] = a;
  bonus[s] = greedy[off + best];
}

__global__ void len_advance_kernel(int32_t* len, const int32_t* by, int32_t inc, int n_seq) {
  const int s = threadIdx.x;
  if (s < n_seq) len[s] += by ? by[s] : inc;
}

}  // namespace tv

using namespace tv;

extern "C" size_t tv_tree_meta_bytes(int32_t n_seq, int32_t n_total) {
  (void)n_seq;
  return n_total > 0 ? meta_bytes(n_total) : 0;
}

extern "C" tv_status tv_tree_prepare(const tv_tree* t, tv_stream stream) {
  if (!tree_ok(t)) return TV_ERR_ARG;
  tree_prepare_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      t->node_off, t->parent, t->meta, t->status, t->n_seq, t->n_total, t->n_max);
  return launch_status();
}

extern "C" tv_status tv_accept_path(const tv_tree* t, const int32_t* tok, const int32_t* greedy, int32_t* path,
                                    int32_t* acc_len, int32_t* bonus, tv_stream stream) {
  if (!tree_ok(t) || !tok || !greedy || !path || !acc_len || !bonus) return TV_ERR_ARG;
  if (!aligned16(tok) || !aligned16(greedy) || !aligned16(path) || !aligned16(acc_len) || !aligned16(bonus))
    return TV_ERR_ALIGN;
  accept_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(tok, greedy, t->meta, t->n_seq, t->n_total,
                                                                       path, acc_len, bonus, t->status);
  return launch_status();
}

extern "C" tv_status tv_len_advance(int32_t* len, const int32_t* by, int32_t inc, int32_t n_seq, tv_stream stream) {
  if (!len || n_seq < 1 || n_seq > TV_MAX_SEQ) return TV_ERR_ARG;
  if (!aligned16(len) || (by && !aligned16(by))) return TV_ERR_ALIGN;
  len_advance_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(len, by, inc, n_seq);
  return launch_status();
}
