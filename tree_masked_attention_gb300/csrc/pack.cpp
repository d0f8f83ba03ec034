// Host packing: sequences -> token trie -> preorder rows, depth positions, subtree
// intervals, compressed nodes and next-token occurrences.
//
// Trie packing (agillm.io), "Step 1 - Store each node once": a token is shared only
// when its whole preceding context is identical, and its position is its depth.
// Tree Training (arXiv 2511.00413) §3.1 eq. 8: DFS serialisation; §3.2 eq. 9:
// depth positions. Claw-R1 "Prefix Tree Merge", "1. build and compress": insert,
// compress single-child chains into nodes, number them in preorder.
//
// The trie is stored as flat arrays with insertion-ordered child lists
// (first_child / next_sibling); a child is looked up by scanning its parent's list, or,
// for a node with many children, through a hash map from (parent, token), so building
// is O(total tokens) and the preorder walk needs no recursion (paths of several
// thousand tokens are common).
#include <algorithm>
#include <cstring>
#include <new>
#include <unordered_map>
#include <vector>

#include "common.h"

struct tree_plan {
  int64_t n_seqs = 0;
  std::vector<int64_t> offsets;     // [n_seqs + 1]
  std::vector<int32_t> tokens;      // copy of the input tokens
  std::vector<int32_t> token_node;  // trie node of every input token
  // trie
  std::vector<int32_t> tok, parent, first_child, last_child, next_sibling, n_child, through, ends;
  int32_t first_root = -1, last_root = -1;
  // preorder
  std::vector<int32_t> order;   // row -> trie node
  std::vector<int32_t> row_of;  // trie node -> row
  std::vector<int32_t> depth;   // trie node -> depth
  std::vector<int32_t> node_start;
  int64_t n_occ = 0, n_roots = 0;
};

namespace {

inline uint64_t edge_key(int32_t parent, int32_t token) {
  return (static_cast<uint64_t>(static_cast<uint32_t>(parent + 1)) << 32) |
         static_cast<uint32_t>(token);
}

// A child is found by scanning its parent's insertion-ordered child list (one compare
// along a chain, a few at a fork); a node with more than kScan children also gets its
// children into a hash map keyed by (parent, token), which serves its later lookups.
constexpr int32_t kScan = 16;

int build(tree_plan& p) {
  const int64_t n_tokens = p.offsets[p.n_seqs];
  std::unordered_map<uint64_t, int32_t> wide;  // children of nodes with > kScan children
  p.token_node.resize(static_cast<size_t>(n_tokens));
  p.tok.reserve(static_cast<size_t>(n_tokens));
  auto kids_of = [&](int32_t node) { return node < 0 ? p.first_root : p.first_child[node]; };
  auto fanout = [&](int32_t node) -> int64_t { return node < 0 ? p.n_roots : p.n_child[node]; };
  auto find_child = [&](int32_t node, int32_t tk) -> int32_t {
    if (fanout(node) > kScan) {
      auto it = wide.find(edge_key(node, tk));
      return it == wide.end() ? -1 : it->second;
    }
    for (int32_t c = kids_of(node); c >= 0; c = p.next_sibling[c])
      if (p.tok[c] == tk) return c;
    return -1;
  };
  for (int64_t k = 0; k < p.n_seqs; ++k) {
    int32_t node = -1;
    for (int64_t t = p.offsets[k]; t < p.offsets[k + 1]; ++t) {
      const int32_t tk = p.tokens[t];
      int32_t c = find_child(node, tk);
      if (c < 0) {
        if (p.tok.size() >= static_cast<size_t>(INT32_MAX))
          return tree::fail(TREE_ERR_SHAPE, "tree_pack_plan: more than 2^31-1 packed rows");
        c = static_cast<int32_t>(p.tok.size());
        p.tok.push_back(tk);
        p.parent.push_back(node);
        p.first_child.push_back(-1);
        p.last_child.push_back(-1);
        p.next_sibling.push_back(-1);
        p.n_child.push_back(0);
        p.through.push_back(0);
        p.ends.push_back(0);
        p.depth.push_back(node < 0 ? 0 : p.depth[node] + 1);
        if (node < 0) {
          if (p.last_root < 0) p.first_root = c; else p.next_sibling[p.last_root] = c;
          p.last_root = c;
          ++p.n_roots;
        } else {
          if (p.last_child[node] < 0) p.first_child[node] = c; else p.next_sibling[p.last_child[node]] = c;
          p.last_child[node] = c;
          ++p.n_child[node];
        }
        const int64_t f = fanout(node);
        if (f == kScan + 1) {  // the node just became wide: index all its children
          for (int32_t s = kids_of(node); s >= 0; s = p.next_sibling[s]) wide.emplace(edge_key(node, p.tok[s]), s);
        } else if (f > kScan + 1) {
          wide.emplace(edge_key(node, tk), c);
        }
      }
      ++p.through[c];
      p.token_node[t] = c;
      node = c;
    }
    if (node >= 0) ++p.ends[node];
    const int64_t len = p.offsets[k + 1] - p.offsets[k];
    if (len > 1) p.n_occ += len - 1;
  }
  if (p.n_occ > INT32_MAX)
    return tree::fail(TREE_ERR_SHAPE, "tree_pack_plan: more than 2^31-1 occurrences");

  // preorder walk over insertion-ordered children (eq. 8)
  const size_t T = p.tok.size();
  p.order.reserve(T);
  p.row_of.assign(T, -1);
  int32_t cur = p.first_root;
  while (cur >= 0) {
    p.row_of[cur] = static_cast<int32_t>(p.order.size());
    p.order.push_back(cur);
    if (p.first_child[cur] >= 0) { cur = p.first_child[cur]; continue; }
    while (cur >= 0 && p.next_sibling[cur] < 0) cur = p.parent[cur];
    if (cur >= 0) cur = p.next_sibling[cur];
  }
  // nodes (chunks): start at roots, below forks and below sequence ends
  for (size_t i = 0; i < T; ++i) {
    const int32_t par = p.parent[p.order[i]];
    if (par < 0 || p.n_child[par] != 1 || p.ends[par] > 0)
      p.node_start.push_back(static_cast<int32_t>(i));
  }
  return TREE_OK;
}

}  // namespace

extern "C" int tree_pack_plan(const int32_t* tokens, const int64_t* seq_offsets, int64_t n_seqs,
                              tree_plan** plan, tree_pack_sizes* sizes) {
  tree::clear_error();
  if (!plan || !sizes || !seq_offsets || n_seqs < 0)
    return tree::fail(TREE_ERR_INVALID_ARG, "tree_pack_plan: null argument or n_seqs < 0");
  *plan = nullptr;
  if (seq_offsets[0] != 0) return tree::fail(TREE_ERR_INVALID_ARG, "tree_pack_plan: seq_offsets[0] != 0");
  for (int64_t k = 0; k < n_seqs; ++k)
    if (seq_offsets[k + 1] < seq_offsets[k])
      return tree::fail(TREE_ERR_INVALID_ARG, "tree_pack_plan: seq_offsets decreases at %lld",
                        static_cast<long long>(k));
  const int64_t n_tokens = seq_offsets[n_seqs];
  if (n_tokens > 0 && !tokens) return tree::fail(TREE_ERR_INVALID_ARG, "tree_pack_plan: tokens is null");
  tree_plan* p = new (std::nothrow) tree_plan();
  if (!p) return tree::fail(TREE_ERR_INVALID_ARG, "tree_pack_plan: out of host memory");
  try {
    p->n_seqs = n_seqs;
    p->offsets.assign(seq_offsets, seq_offsets + n_seqs + 1);
    p->tokens.assign(tokens, tokens + n_tokens);
    int st = build(*p);
    if (st != TREE_OK) { delete p; return st; }
  } catch (const std::bad_alloc&) {
    delete p;
    return tree::fail(TREE_ERR_INVALID_ARG, "tree_pack_plan: out of host memory");
  }
  sizes->T = static_cast<int64_t>(p->order.size());
  sizes->n_nodes = static_cast<int64_t>(p->node_start.size());
  sizes->n_occ = p->n_occ;
  sizes->n_roots = p->n_roots;
  sizes->n_tokens = n_tokens;
  *plan = p;
  return TREE_OK;
}

extern "C" int tree_pack_emit(const tree_plan* plan, const float* seq_weights, const tree_pack_out* out) {
  tree::clear_error();
  if (!plan || !out) return tree::fail(TREE_ERR_INVALID_ARG, "tree_pack_emit: null argument");
  const tree_plan& p = *plan;
  const int32_t T = static_cast<int32_t>(p.order.size());
  const int32_t n_nodes = static_cast<int32_t>(p.node_start.size());
  try {
    // parent rows and subtree ends (children follow their parent in preorder, so a
    // reverse sweep accumulates subtree sizes)
    std::vector<int32_t> prow(T), size(T, 1);
    for (int32_t i = 0; i < T; ++i) {
      const int32_t par = p.parent[p.order[i]];
      prow[i] = par < 0 ? -1 : p.row_of[par];
    }
    for (int32_t i = T - 1; i >= 0; --i)
      if (prow[i] >= 0) size[prow[i]] += size[i];
    std::vector<int32_t> node_of(out->node_of_token || out->node_parent ? T : 0);
    for (int32_t c = 0; c < n_nodes && !node_of.empty(); ++c) {
      const int32_t s = p.node_start[c], e = c + 1 < n_nodes ? p.node_start[c + 1] : T;
      for (int32_t i = s; i < e; ++i) node_of[i] = c;
    }
    for (int32_t i = 0; i < T; ++i) {
      const int32_t n = p.order[i];
      if (out->packed_ids) out->packed_ids[i] = p.tok[n];
      if (out->position_ids) out->position_ids[i] = p.depth[n];
      if (out->subtree_end) out->subtree_end[i] = i + size[i] - 1;
      if (out->path_count) out->path_count[i] = p.through[n];
      if (out->parent_row) out->parent_row[i] = prow[i];
      if (out->node_of_token) out->node_of_token[i] = node_of[i];
    }
    for (int32_t c = 0; c < n_nodes; ++c) {
      const int32_t s = p.node_start[c];
      if (out->node_start) out->node_start[c] = s;
      if (out->node_end) out->node_end[c] = (c + 1 < n_nodes ? p.node_start[c + 1] : T) - 1;
      if (out->node_parent) out->node_parent[c] = prow[s] < 0 ? -1 : node_of[prow[s]];
    }
    const int64_t n_tokens = p.offsets[p.n_seqs];
    if (out->token_rows)
      for (int64_t t = 0; t < n_tokens; ++t) out->token_rows[t] = p.row_of[p.token_node[t]];
    // occurrences, sequence-major; CSR by source row through a stable counting sort
    if (!out->occ_source_rows && !out->occ_targets && !out->occ_seq && !out->occ_weights && !out->occ_row_ptr &&
        !out->occ_perm)
      return TREE_OK;
    std::vector<int32_t> count(static_cast<size_t>(T) + 1, 0);
    int32_t o = 0;
    for (int64_t k = 0; k < p.n_seqs; ++k) {
      const float w = seq_weights ? seq_weights[k] : 1.0f;
      for (int64_t t = p.offsets[k]; t + 1 < p.offsets[k + 1]; ++t, ++o) {
        const int32_t r = p.row_of[p.token_node[t]];
        if (out->occ_source_rows) out->occ_source_rows[o] = r;
        if (out->occ_targets) out->occ_targets[o] = p.tokens[t + 1];
        if (out->occ_seq) out->occ_seq[o] = static_cast<int32_t>(k);
        if (out->occ_weights) out->occ_weights[o] = w;
        ++count[r + 1];
      }
    }
    for (int32_t r = 0; r < T; ++r) count[r + 1] += count[r];
    if (out->occ_row_ptr) std::memcpy(out->occ_row_ptr, count.data(), sizeof(int32_t) * (T + 1));
    if (out->occ_perm) {
      std::vector<int32_t> fill(count.begin(), count.end() - 1);
      o = 0;
      for (int64_t k = 0; k < p.n_seqs; ++k)
        for (int64_t t = p.offsets[k]; t + 1 < p.offsets[k + 1]; ++t, ++o)
          out->occ_perm[fill[p.row_of[p.token_node[t]]]++] = o;
    }
  } catch (const std::bad_alloc&) {
    return tree::fail(TREE_ERR_INVALID_ARG, "tree_pack_emit: out of host memory");
  }
  return TREE_OK;
}

extern "C" void tree_plan_free(tree_plan* plan) { delete plan; }

extern "C" int tree_validate_subtree_end(const int32_t* end, int64_t T) {
  tree::clear_error();
  if (T < 0 || (T > 0 && !end)) return tree::fail(TREE_ERR_INVALID_ARG, "tree_validate_subtree_end: bad arguments");
  std::vector<int64_t> open;  // ends of the intervals enclosing the current row
  for (int64_t i = 0; i < T; ++i) {
    const int64_t e = end[i];
    if (e < i || e >= T)
      return tree::fail(TREE_ERR_INVALID_ARG, "subtree_end[%lld] = %lld outside [i, T)",
                        static_cast<long long>(i), static_cast<long long>(e));
    while (!open.empty() && open.back() < i) open.pop_back();
    if (!open.empty() && e > open.back())
      return tree::fail(TREE_ERR_INVALID_ARG, "subtree of row %lld (end %lld) leaves its parent's (end %lld)",
                        static_cast<long long>(i), static_cast<long long>(e),
                        static_cast<long long>(open.back()));
    open.push_back(e);
  }
  return TREE_OK;
}
