// SWA component of the radix prefix cache (host C++).
//
// Method: "SWA in SGLang" design note, section "prefix cache: tombstones and
// the window hit rule": a cached node may keep its full KV after its SWA KV
// was released (a tombstone); a match may end only where the W tokens before
// it are live (the match falls back to the last such position); two LRU
// lists (full eviction deletes leaves, SWA eviction turns nodes into
// tombstones, and a leaf may not be a tombstone); the full lock reaches the
// root while the SWA lock covers only the last W tokens; insert puts
// [0, swa_evicted) in as a tombstone prefix and revives tombstones the new
// request has SWA KV for.  Readings (whole pages, splitting at the match end,
// time stamps, duplicate release, LRU ties by creation order, locks returning
// their SWA span) are stated at the declarations in include/swa.h.
//
// The tree holds full slots on the host and never touches the device: every
// operation reports the slots whose KV must go back (full + SWA through
// swa_free, or SWA only through swa_free_swa) with their page counts, and the
// caller issues those calls on its stream.
#include <stdint.h>

#include <algorithm>
#include <map>
#include <memory>
#include <new>
#include <set>
#include <utility>
#include <vector>

#include "swa.h"

namespace {

struct Node {
  std::vector<int32_t> key;
  std::vector<int64_t> full;
  bool tomb = false;
  std::map<std::vector<int32_t>, int64_t> children;   // first page -> node id
  int64_t parent = -1;
  int64_t full_lock = 0, swa_lock = 0;
  uint64_t t_full = 0, t_swa = 0;
  int64_t id = 0;
};

}  // namespace

struct swa_radix {
  int64_t ps = 1;
  int64_t W = 0;
  uint64_t clock = 0;
  std::vector<std::unique_ptr<Node>> nodes;            // by id; null once deleted
  std::set<std::pair<uint64_t, int64_t>> lru_full, lru_swa;   // (stamp, id) of every non-root node
  std::vector<int64_t> rel_full, rel_swa;               // releases since the last read
  int64_t rel_full_live = 0;                            // tokens of rel_full that had SWA KV
  std::vector<int64_t> out_full, out_swa;               // handed out by swa_radix_releases
  int64_t cached = 0, live = 0;

  Node *node(int64_t id) { return id >= 0 && id < (int64_t)nodes.size() ? nodes[id].get() : nullptr; }
  std::vector<int32_t> page(const std::vector<int32_t> &k, size_t i) const {
    return std::vector<int32_t>(k.begin() + i, k.begin() + i + ps);
  }
  void stamp(Node *n, uint64_t t) {
    if (n->id == 0) return;
    lru_full.erase({n->t_full, n->id});
    lru_swa.erase({n->t_swa, n->id});
    n->t_full = n->t_swa = t;
    lru_full.insert({t, n->id});
    lru_swa.insert({t, n->id});
  }
  Node *make(std::vector<int32_t> key, std::vector<int64_t> full, bool tomb, Node *parent,
             uint64_t tf, uint64_t ts) {
    auto up = std::make_unique<Node>();
    Node *n = up.get();
    n->id = (int64_t)nodes.size();
    n->key = std::move(key);
    n->full = std::move(full);
    n->tomb = tomb;
    n->parent = parent->id;
    n->t_full = tf;
    n->t_swa = ts;
    nodes.push_back(std::move(up));
    parent->children[page(n->key, 0)] = n->id;
    lru_full.insert({tf, n->id});
    lru_swa.insert({ts, n->id});
    cached += (int64_t)n->key.size();
    if (!tomb) live += (int64_t)n->key.size();
    return n;
  }
  // node keeps key[k:]; a new parent takes key[:k] with the same flags,
  // stamps and lock counts.
  Node *split(Node *n, size_t k) {
    Node *parent = node(n->parent);
    std::vector<int32_t> tk(n->key.begin(), n->key.begin() + k);
    std::vector<int64_t> tf(n->full.begin(), n->full.begin() + k);
    cached -= (int64_t)k;                 // make() adds them back
    if (!n->tomb) live -= (int64_t)k;
    Node *top = make(std::move(tk), std::move(tf), n->tomb, parent, n->t_full, n->t_swa);
    top->full_lock = n->full_lock;
    top->swa_lock = n->swa_lock;
    n->key.erase(n->key.begin(), n->key.begin() + k);
    n->full.erase(n->full.begin(), n->full.begin() + k);
    n->parent = top->id;
    top->children[page(n->key, 0)] = n->id;
    return top;
  }
  // Slots v[a, b) go back; `with_swa` of them (full releases) still map an SWA slot.
  void release(const std::vector<int64_t> &v, size_t a, size_t b, bool swa_only, size_t with_swa) {
    auto &dst = swa_only ? rel_swa : rel_full;
    dst.insert(dst.end(), v.begin() + a, v.begin() + b);
    if (!swa_only) rel_full_live += (int64_t)with_swa;
  }
  void erase(Node *n) {
    Node *parent = node(n->parent);
    parent->children.erase(page(n->key, 0));
    lru_full.erase({n->t_full, n->id});
    lru_swa.erase({n->t_swa, n->id});
    cached -= (int64_t)n->key.size();
    if (!n->tomb) live -= (int64_t)n->key.size();
    nodes[n->id].reset();
  }
  int64_t drop_leaf(Node *leaf) {
    int64_t freed = (int64_t)leaf->key.size();
    release(leaf->full, 0, leaf->full.size(), false, leaf->tomb ? 0 : leaf->full.size());
    Node *parent = node(leaf->parent);
    erase(leaf);
    while (parent->id != 0 && parent->children.empty() && parent->tomb) {
      freed += (int64_t)parent->key.size();
      release(parent->full, 0, parent->full.size(), false, 0);
      Node *up = node(parent->parent);
      erase(parent);
      parent = up;
    }
    return freed;
  }
  // tokens of `key` (length n) that the child of `nd` starting at pos matches
  size_t common(const Node *child, const std::vector<int32_t> &key, size_t pos, size_t n) const {
    size_t c = 0;
    while (c < child->key.size() && pos + c < n &&
           std::equal(child->key.begin() + c, child->key.begin() + c + ps, key.begin() + pos + c))
      c += ps;
    return c;
  }
  Node *child_of(Node *nd, const std::vector<int32_t> &key, size_t pos) {
    auto it = nd->children.find(page(key, pos));
    return it == nd->children.end() ? nullptr : node(it->second);
  }
};

extern "C" {

swa_status swa_radix_create(int32_t page_size, int32_t window, swa_radix **out) {
  if (!out || page_size < 1 || window < 0) return SWA_ERR_INVALID;
  swa_radix *t = new (std::nothrow) swa_radix();
  if (!t) return SWA_ERR_INVALID;
  t->ps = page_size;
  t->W = window;
  auto root = std::make_unique<Node>();
  root->id = 0;
  t->nodes.push_back(std::move(root));
  *out = t;
  return SWA_OK;
}

void swa_radix_destroy(swa_radix *t) { delete t; }

swa_status swa_radix_match(swa_radix *t, const int32_t *tokens, int64_t n_tok, int64_t *e_out,
                           int64_t *slots_out, int64_t *node_out) {
  if (!t || n_tok < 0 || (n_tok > 0 && !tokens) || !e_out || !node_out) return SWA_ERR_INVALID;
  const size_t n = (size_t)(n_tok / t->ps * t->ps);
  std::vector<int32_t> key(tokens, tokens + n);
  const uint64_t now = ++t->clock;
  std::vector<std::pair<Node *, size_t>> path;
  Node *nd = t->node(0);
  size_t pos = 0;
  while (pos < n) {
    Node *ch = t->child_of(nd, key, pos);
    if (!ch) break;
    const size_t c = t->common(ch, key, pos, n);
    path.push_back({ch, c});
    pos += c;
    if (c < ch->key.size()) break;
    nd = ch;
  }
  // Usable ends: the run of live tokens before e reaches W, or the root.
  std::vector<char> ok(pos + 1, 0);
  ok[0] = 1;
  int64_t run = 0;
  bool at_root = true;
  size_t i = 0;
  for (auto &pc : path)
    for (size_t j = 0; j < pc.second; ++j, ++i) {
      if (pc.first->tomb) {
        run = 0;
        at_root = false;
      } else {
        ++run;
      }
      ok[i + 1] = (run >= t->W || at_root) ? 1 : 0;
    }
  size_t e = pos;
  while (e > 0 && !ok[e]) e -= t->ps;
  size_t acc = 0, w = 0;
  Node *end = t->node(0);
  for (auto &pc : path) {
    if (acc >= e) break;
    Node *m = pc.first;
    const size_t take = std::min(m->key.size(), e - acc);
    if (take < m->key.size()) m = t->split(m, take);
    if (slots_out)
      for (int64_t s : m->full) slots_out[w++] = s;
    t->stamp(m, now);
    acc += take;
    end = m;
  }
  *e_out = (int64_t)e;
  *node_out = end->id;
  return SWA_OK;
}

swa_status swa_radix_lock(swa_radix *t, int64_t id, int64_t *swa_span) {
  if (!t || !swa_span || !t->node(id)) return SWA_ERR_INVALID;
  int64_t acc = 0, span = 0;
  for (Node *nd = t->node(id); nd->id != 0; nd = t->node(nd->parent)) {
    nd->full_lock += 1;
    if (acc < t->W) {
      nd->swa_lock += 1;
      span = acc + (int64_t)nd->key.size();
    }
    acc += (int64_t)nd->key.size();
  }
  *swa_span = span;
  return SWA_OK;
}

swa_status swa_radix_unlock(swa_radix *t, int64_t id, int64_t swa_span) {
  if (!t || !t->node(id)) return SWA_ERR_INVALID;
  int64_t acc = 0;
  for (Node *nd = t->node(id); nd->id != 0; nd = t->node(nd->parent)) {
    if (nd->full_lock < 1 || (acc < swa_span && nd->swa_lock < 1)) return SWA_ERR_INVALID;
    acc += (int64_t)nd->key.size();
  }
  acc = 0;
  for (Node *nd = t->node(id); nd->id != 0; nd = t->node(nd->parent)) {
    nd->full_lock -= 1;
    if (acc < swa_span) nd->swa_lock -= 1;
    acc += (int64_t)nd->key.size();
  }
  return SWA_OK;
}

swa_status swa_radix_insert(swa_radix *t, const int32_t *tokens, int64_t n_tok,
                            const int64_t *slots, int64_t swa_evicted) {
  if (!t || n_tok < 0 || (n_tok > 0 && (!tokens || !slots)) || swa_evicted < 0 ||
      swa_evicted % t->ps)
    return SWA_ERR_INVALID;
  const size_t n = (size_t)(n_tok / t->ps * t->ps);
  std::vector<int32_t> key(tokens, tokens + n);
  std::vector<int64_t> val(slots, slots + n);
  const size_t ev = std::min((size_t)swa_evicted, n);
  const uint64_t now = ++t->clock;
  Node *nd = t->node(0);
  size_t pos = 0;
  while (pos < n) {
    Node *ch = t->child_of(nd, key, pos);
    if (!ch) break;
    const size_t c = t->common(ch, key, pos, n);
    if (c < ch->key.size()) ch = t->split(ch, c);
    if (ch->tomb && pos < ev && ev < pos + c) {   // request has SWA KV from ev on
      t->split(ch, ev - pos);
      continue;
    }
    if (std::equal(ch->full.begin(), ch->full.end(), val.begin() + pos)) {
      // the request's prefix came from this node: nothing to release
    } else if (ch->tomb && pos >= ev) {            // revive with the request's slots
      t->release(ch->full, 0, ch->full.size(), false, 0);
      ch->full.assign(val.begin() + pos, val.begin() + pos + c);
      ch->tomb = false;
      t->live += (int64_t)c;
    } else {                                       // duplicate of cached tokens
      t->release(val, pos, pos + c, false, pos + c > std::max(pos, ev) ? pos + c - std::max(pos, ev) : 0);
    }
    t->stamp(ch, now);
    nd = ch;
    pos += c;
  }
  if (pos < n) {
    if (pos < ev) {
      if (ev < n) {                                // tombstone only ahead of live tokens
        nd = t->make(std::vector<int32_t>(key.begin() + pos, key.begin() + ev),
                     std::vector<int64_t>(val.begin() + pos, val.begin() + ev), true, nd, now, now);
        pos = ev;
      } else {
        t->release(val, pos, n, false, 0);
        return SWA_OK;
      }
    }
    t->make(std::vector<int32_t>(key.begin() + pos, key.end()),
            std::vector<int64_t>(val.begin() + pos, val.end()), false, nd, now, now);
  }
  return SWA_OK;
}

swa_status swa_radix_evict(swa_radix *t, int32_t swa_only, int64_t n_tokens, int64_t *freed_out) {
  if (!t || n_tokens < 0) return SWA_ERR_INVALID;
  int64_t freed = 0;
  while (freed < n_tokens) {
    Node *pick = nullptr;
    if (swa_only) {
      for (auto &p : t->lru_swa) {
        Node *m = t->node(p.second);
        if (!m->tomb && m->swa_lock == 0 && (!m->children.empty() || m->full_lock == 0)) {
          pick = m;
          break;
        }
      }
      if (!pick) break;
      freed += (int64_t)pick->key.size();
      if (!pick->children.empty()) {
        t->release(pick->full, 0, pick->full.size(), true, 0);
        pick->tomb = true;
        t->live -= (int64_t)pick->key.size();
      } else {
        t->drop_leaf(pick);
      }
    } else {
      for (auto &p : t->lru_full) {
        Node *m = t->node(p.second);
        if (m->children.empty() && m->full_lock == 0) {
          pick = m;
          break;
        }
      }
      if (!pick) break;
      freed += t->drop_leaf(pick);
    }
  }
  if (freed_out) *freed_out = freed;
  return SWA_OK;
}

swa_status swa_radix_releases(swa_radix *t, const int64_t **full, int64_t *n_full,
                              int64_t *n_full_live, const int64_t **swa, int64_t *n_swa) {
  if (!t || !full || !n_full || !n_full_live || !swa || !n_swa) return SWA_ERR_INVALID;
  t->out_full.swap(t->rel_full);
  t->out_swa.swap(t->rel_swa);
  t->rel_full.clear();
  t->rel_swa.clear();
  *full = t->out_full.data();
  *n_full = (int64_t)t->out_full.size();
  *n_full_live = t->rel_full_live;
  t->rel_full_live = 0;
  *swa = t->out_swa.data();
  *n_swa = (int64_t)t->out_swa.size();
  return SWA_OK;
}

swa_status swa_radix_sizes(const swa_radix *t, int64_t *cached_tokens, int64_t *live_tokens,
                           int64_t *nodes) {
  if (!t || !cached_tokens || !live_tokens || !nodes) return SWA_ERR_INVALID;
  *cached_tokens = t->cached;
  *live_tokens = t->live;
  int64_t c = 0;
  for (auto &p : t->nodes) c += p ? 1 : 0;
  *nodes = c - 1;
  return SWA_OK;
}

}  // extern "C"
