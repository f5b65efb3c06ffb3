// Draft-tree preparation, the accept walk and length bookkeeping.
//
// Tree preparation derives, per node, the depth, the ancestor-or-self bitmask
// (the tree mask of the merged draft tree, "One request, end to end" 2.6),
// the ancestor at every depth (the rows a node attends to past the context)
// and the traversal order of the recurrent layers.  One warp per sequence;
// lane i owns nodes i and i + 32, and every table comes from walking at most
// 15 parent links.
//
// Recurrent traversal.  Every node's Gated DeltaNet state is its parent's
// state advanced by one token, so a depth-first walk needs the parent's state
// only until its last child starts.  Leaves never advance the state (only
// their outputs are needed), so the children of a node are visited leaves
// first, then the non-leaf children lightest subtree first and the heaviest
// last.  A node with two or more non-leaf children saves its state in a slot
// while its light non-leaf subtrees run; the heaviest continues from the slot
// with the slot released.  A save at slot level l happens inside l nested
// light non-leaf subtrees, each at most half of the enclosing subtree, and a
// saving node has at least five nodes below and including it, so a tree of n
// nodes needs at most floor(log2(n / 5)) + 1 slots: 4 for 64 nodes.  The order
// never changes any node's arithmetic: each state is exactly one step from its
// parent's.
//
// Segments.  The walk is cut into runs of visits that neither restore nor
// save a state inside: a run starts at a visit whose parent state comes from
// a slot and ends after a visit whose state must be saved, so a kernel
// walking the tree handles slots only between runs and runs the visits of a
// run without branches.
#include "common.cuh"
#include "host.hpp"

namespace tv {

// Order among the children of one parent: leaves (0), light non-leaf (1), the
// heaviest non-leaf child (2); ties by index.
__device__ __forceinline__ int child_class(int c, const int* nch, const int* heavy, const int* par) {
  return nch[c] == 0 ? 0 : (heavy[par[c]] == c ? 2 : 1);
}

__device__ __forceinline__ void tree_invalid(MetaView& mv, int s, int off, int32_t* status) {
  set_status(status, TV_ERR_TREE);
  mv.seq[s] = SeqInfo{0, off, 0, 0, 0, {0, 0, 0}};
}

__global__ void __launch_bounds__(32) tree_prepare_kernel(const int32_t* __restrict__ node_off,
                                                          const int32_t* __restrict__ parent, void* meta,
                                                          int32_t* status, int n_seq, int n_total, int n_max) {
  pdl_wait();  // the previous round's calls read the tables this kernel rewrites
  const int s = blockIdx.x;
  const int lane = threadIdx.x;
  __shared__ int par[TV_MAX_NODES], nch[TV_MAX_NODES], nnl[TV_MAX_NODES], size[TV_MAX_NODES];
  __shared__ int hkey[TV_MAX_NODES], heavy[TV_MAX_NODES], rel[TV_MAX_NODES], first_light[TV_MAX_NODES];
  __shared__ int vsrc[TV_MAX_NODES], vsave[TV_MAX_NODES];  // the walk's slot use, in visit order
  MetaView mv = meta_view(meta, n_total);
  const int off = node_off[s];
  const int end = node_off[s + 1];
  const int n = end - off;
  const bool ok = off >= 0 && end <= n_total && n >= 1 && n <= n_max && n <= TV_MAX_NODES &&
                  (s > 0 || off == 0) && (s < n_seq - 1 || end == n_total);
  if (!ok) {
    if (lane == 0) tree_invalid(mv, s, off, status);
    return;
  }
  bool good = true;
  for (int i = lane; i < n; i += 32) {
    const int p = parent[off + i];
    good = good && (i == 0 ? p == -1 : (p >= 0 && p < i));
    par[i] = (i == 0 || !(p >= 0 && p < i)) ? -1 : p;
    nch[i] = 0;
    nnl[i] = 0;
    size[i] = 1;
    hkey[i] = -1;
    first_light[i] = 1 << 30;
  }
  if (!__all_sync(0xffffffffu, good)) {
    if (lane == 0) tree_invalid(mv, s, off, status);
    return;
  }
  __syncwarp();
  // depth, ancestor bitmask, ancestor at every depth; subtree sizes; child counts
  int my_depth = 0;
  for (int i = lane; i < n; i += 32) {
    int d = -1;
    uint64_t mask = 0;
    for (int j = i; j != -1; j = par[j]) {
      mask |= 1ull << j;
      d++;
    }
    if (d >= TV_MAX_PATH) {
      good = false;
      continue;
    }
    my_depth = d > my_depth ? d : my_depth;
    mv.anc[off + i] = mask;
    mv.depth[off + i] = d;
    int8_t* row = mv.anc_at + static_cast<size_t>(off + i) * TV_MAX_PATH;
    int e = d;
    for (int j = i; j != -1; j = par[j], e--) row[e] = static_cast<int8_t>(j);
    for (int x = d + 1; x < TV_MAX_PATH; x++) row[x] = -1;
    for (int j = par[i]; j != -1; j = par[j]) atomicAdd(&size[j], 1);
    if (i > 0) atomicAdd(&nch[par[i]], 1);
  }
  if (!__all_sync(0xffffffffu, good)) {
    if (lane == 0) tree_invalid(mv, s, off, status);
    return;
  }
  __syncwarp();
  // non-leaf children and the heaviest of them (largest subtree, lowest index)
  for (int i = lane; i < n; i += 32) {
    if (i > 0 && nch[i] > 0) {
      atomicAdd(&nnl[par[i]], 1);
      atomicMax(&hkey[par[i]], (size[i] << 8) | (255 - i));
    }
  }
  __syncwarp();
  for (int i = lane; i < n; i += 32) heavy[i] = hkey[i] < 0 ? -1 : 255 - (hkey[i] & 255);
  __syncwarp();
  for (int i = lane; i < n; i += 32)
    if (i > 0 && child_class(i, nch, heavy, par) == 1) atomicMin(&first_light[par[i]], i);
  // offset of each node within its parent's subtree: 1 + sizes of the siblings before it
  for (int i = lane; i < n; i += 32) {
    int r = 0;
    if (i > 0) {
      const int p = par[i];
      const int ci = child_class(i, nch, heavy, par);
      r = 1;
      for (int j = p + 1; j < n; j++) {
        if (par[j] != p || j == i) continue;
        const int cj = child_class(j, nch, heavy, par);
        if (cj < ci || (cj == ci && j < i)) r += size[j];
      }
    }
    rel[i] = r;
  }
  __syncwarp();
  // preorder position, slot levels and the traversal entry of every node
  int my_slot = -1;
  for (int i = lane; i < n; i += 32) {
    int pos = 0, lv = 0, last_edge_light = 0;
    for (int j = i; j > 0; j = par[j]) {
      pos += rel[j];
      const int light = (nnl[par[j]] >= 2 && child_class(j, nch, heavy, par) == 1) ? 1 : 0;
      if (j == i) last_edge_light = light;
      lv += light;
    }
    const int lv_parent = lv - last_edge_light;
    int src = 0;
    if (i > 0) {
      const int p = par[i];
      const int ci = child_class(i, nch, heavy, par);
      const bool from_registers = ci == 0 || nnl[p] < 2 || (ci == 1 && first_light[p] == i);
      src = from_registers ? 0 : 1 + lv_parent;
    }
    int save = 0;
    if (nnl[i] >= 2) {
      save = 1 + lv;
      my_slot = lv > my_slot ? lv : my_slot;
    }
    if (lv >= kMaxSlots) good = false;
    mv.sched[off + pos] = visit_encode(i, nch[i] > 0 ? 1 : 0);
    vsrc[pos] = src;
    vsave[pos] = save;
  }
  if (!__all_sync(0xffffffffu, good)) {
    if (lane == 0) tree_invalid(mv, s, off, status);
    return;
  }
  __syncwarp();
  // cut the walk into segments (one lane; at most 64 visits)
  int n_seg = 0;
  if (lane == 0) {
    int first = 0;
    for (int v = 1; v <= n; v++) {
      if (v == n || vsrc[v] != 0 || vsave[v - 1] != 0) {
        mv.seg[off + n_seg] = seg_encode(first, v - first, vsrc[first], vsave[v - 1]);
        n_seg++;
        first = v;
      }
    }
  }
  n_seg = __shfl_sync(0xffffffffu, n_seg, 0);
  for (int o = 16; o >= 1; o >>= 1) {
    my_depth = max(my_depth, __shfl_xor_sync(0xffffffffu, my_depth, o));
    my_slot = max(my_slot, __shfl_xor_sync(0xffffffffu, my_slot, o));
  }
  if (lane == 0) mv.seq[s] = SeqInfo{n, off, my_depth, my_slot + 1, n_seg, {0, 0, 0}};
}

// Longest agreeing path plus one token ("One request, end to end" 2.6).
// One warp per sequence: a node agrees when every edge on its root path
// carries the target's greedy token at the edge's parent; the deepest agreeing
// node wins, lowest index among equally deep ones.
__global__ void __launch_bounds__(32) accept_kernel(const int32_t* __restrict__ tok,
                                                    const int32_t* __restrict__ greedy, const void* meta,
                                                    int n_total, int32_t* path, int32_t* acc_len, int32_t* bonus,
                                                    int32_t* status) {
  pdl_wait();
  const int s = blockIdx.x;
  const int lane = threadIdx.x;
  int32_t* prow = path + s * TV_MAX_PATH;
  if (status_bad(status)) {
    if (lane < TV_MAX_PATH) prow[lane] = -1;
    if (lane == 0) {
      acc_len[s] = 0;
      bonus[s] = -1;
    }
    return;
  }
  MetaView mv = meta_view(const_cast<void*>(meta), n_total);
  const SeqInfo info = mv.seq[s];
  const int n = info.n, off = info.off;
  int key = -1;
  for (int i = lane; i < n; i += 32) {
    const int d = mv.depth[off + i];
    const int8_t* row = mv.anc_at + static_cast<size_t>(off + i) * TV_MAX_PATH;
    bool agree = true;
    for (int e = 1; e <= d; e++) agree = agree && tok[off + row[e]] == greedy[off + row[e - 1]];
    if (agree) key = max(key, (d << 8) | (255 - i));
  }
  for (int o = 16; o >= 1; o >>= 1) key = max(key, __shfl_xor_sync(0xffffffffu, key, o));
  const int best = 255 - (key & 255);
  const int a = (key >> 8) + 1;
  const int8_t* arow = mv.anc_at + static_cast<size_t>(off + best) * TV_MAX_PATH;
  if (lane < TV_MAX_PATH) prow[lane] = lane < a ? arow[lane] : -1;
  if (lane == 0) {
    acc_len[s] = a;
    bonus[s] = greedy[off + best];
  }
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
  launch_k(tree_overlap(t), tree_prepare_kernel, dim3(t->n_seq), dim3(32), 0, reinterpret_cast<cudaStream_t>(stream),
           t->node_off, t->parent, t->meta, t->status, t->n_seq, t->n_total, t->n_max);
  return launch_status();
}

extern "C" tv_status tv_accept_path(const tv_tree* t, const int32_t* tok, const int32_t* greedy, int32_t* path,
                                    int32_t* acc_len, int32_t* bonus, tv_stream stream) {
  if (!tree_ok(t) || !tok || !greedy || !path || !acc_len || !bonus) return TV_ERR_ARG;
  if (!aligned16(tok) || !aligned16(greedy) || !aligned16(path) || !aligned16(acc_len) || !aligned16(bonus))
    return TV_ERR_ALIGN;
  launch_k(tree_overlap(t), accept_kernel, dim3(t->n_seq), dim3(32), 0, reinterpret_cast<cudaStream_t>(stream), tok,
           greedy, static_cast<const void*>(t->meta), t->n_total, path, acc_len, bonus, t->status);
  return launch_status();
}

extern "C" tv_status tv_len_advance(int32_t* len, const int32_t* by, int32_t inc, int32_t n_seq, tv_stream stream) {
  if (!len || n_seq < 1 || n_seq > TV_MAX_SEQ) return TV_ERR_ARG;
  if (!aligned16(len) || (by && !aligned16(by))) return TV_ERR_ALIGN;
  len_advance_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(len, by, inc, n_seq);
  return launch_status();
}
