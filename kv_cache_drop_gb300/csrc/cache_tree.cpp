// Extended radix tree of cache histories and drop-aware eviction (paper
// review page section 4.2 "AKV serving": a radix tree whose paths carry the
// cache-operation history next to the tokens -- drop nodes record which
// entries were removed, a repos opens a branch with re-numbered positions --
// and an eviction policy that frees physical KV only when no running
// computation uses it, dropped entries before finished requests' entries,
// keeping tree nodes as empty placeholders and treating each position
// version separately; section 3.4 / Figure 5: the same surviving tokens can
// have different KV when the operations happened in a different order).
//
// A request history is its messages (token ids) with the operations listed
// after each message (operate-after: the drops of a boundary as a set, then
// an optional repos).  The tree interleaves message nodes (edge label = the
// message's token ids) and operation nodes (edge label = the boundary's
// drop set and repos flag): a message node stands for the KV of that
// message computed after exactly the history on its path, so two requests
// share it iff their histories agree up to it.
//
// Storage units: a message node's own KV (at the positions it was computed
// with), and at every repos node one re-rotated copy of each message alive
// there (the new position version).  Each unit is resident or evicted,
// pinned by the running requests whose active cache uses it (the pin count
// is the reference count of that position version), and marked dropped
// when the latest request using it dropped it.
//
// Pool trees (akv_tree_create_pool) also manage the token slots of a
// page-size-1 KV pool (the system README: drop and repos support page size 1
// only): a resident unit owns one slot per token, eviction returns its slots
// to the free list, an insert takes slots for the units it makes resident
// (lowest free slots first), evicting unpinned units in the same drop-aware
// order when the free list is short, and a running request can hold extra
// slots for its decode appends until it finishes.
#include <algorithm>
#include <cstdint>
#include <iterator>
#include <map>
#include <memory>
#include <vector>

#include "akv_internal.h"

using namespace akv;

struct akv_tree;

namespace {

struct Unit {  // one storage unit: the KV of one message at one position version
  int64_t tokens = 0;
  bool resident = false;
  bool dropped = false;
  int pins = 0;
  uint64_t last_use = 0;  // insert count of the latest request holding it
  uint64_t seq = 0;       // creation order (ties in eviction order)
  bool busy = false;      // on the path of the insert in progress (not evictable by it)
  std::vector<int32_t> slots;  // pool trees: one pool slot per token while resident
};

struct Node {
  enum Kind { kRoot, kMsg, kOps } kind = kRoot;
  std::vector<int32_t> tokens;       // kMsg: the message's token ids
  std::vector<int32_t> drops;        // kOps: sorted dropped message ordinals
  bool repos = false;                // kOps
  Node *parent = nullptr;
  std::vector<std::unique_ptr<Node>> children;
  Unit own;                          // kMsg: the message's KV as computed
  std::map<const Node *, Unit> ver;  // kOps with repos: re-rotated copies, by message node
};

// One boundary's operations in canonical form.
struct OpSet {
  std::vector<int32_t> drops;
  bool repos = false;
  bool empty() const { return drops.empty() && !repos; }
};

std::vector<OpSet> op_sets(const akv_oplog *o) {
  std::vector<OpSet> ops(o->n_msgs);
  for (int i = 0; i < o->n_drops; ++i) ops[o->drop_after[i]].drops.push_back(o->drop_target[i]);
  for (int i = 0; i < o->n_repos; ++i) ops[o->repos_after[i]].repos = true;
  for (OpSet &s : ops) {
    std::sort(s.drops.begin(), s.drops.end());
    s.drops.erase(std::unique(s.drops.begin(), s.drops.end()), s.drops.end());
  }
  return ops;
}

Node *find_msg(Node *n, const int32_t *tok, int64_t len) {
  for (auto &c : n->children)
    if (c->kind == Node::kMsg && (int64_t)c->tokens.size() == len &&
        std::equal(c->tokens.begin(), c->tokens.end(), tok))
      return c.get();
  return nullptr;
}

Node *find_ops(Node *n, const OpSet &s) {
  for (auto &c : n->children)
    if (c->kind == Node::kOps && c->repos == s.repos && c->drops == s.drops) return c.get();
  return nullptr;
}

// Replay of a history's cache state: alive flags and, per version, the
// position of each message's first token (positions inside a message are
// consecutive in every version).
struct Replay {
  std::vector<std::vector<char>> alive_before;  // [m][j]: j alive when message m starts
  std::vector<char> alive_end;
  std::vector<int> ver_of;                      // version current when message m was appended
  std::vector<std::vector<int64_t>> first_pos;  // [v][j], -1 if j not in version v
  int n_ver = 1;
};

Replay replay(const akv_oplog *o, const std::vector<OpSet> &ops) {
  const int n = o->n_msgs;
  Replay r;
  std::vector<char> alive(n, 0);
  r.alive_before.assign(n, {});
  r.ver_of.assign(n, 0);
  r.first_pos.assign(1, std::vector<int64_t>(n, -1));
  int64_t next = 0;
  int v = 0;
  for (int m = 0; m < n; ++m) {
    r.alive_before[m] = alive;
    r.ver_of[m] = v;
    r.first_pos[v][m] = next;
    next += o->msg_start[m + 1] - o->msg_start[m];
    alive[m] = 1;
    for (int j : ops[m].drops) alive[j] = 0;
    if (ops[m].repos) {
      ++v;
      r.first_pos.emplace_back(n, -1);
      int64_t p = 0;
      for (int j = 0; j <= m; ++j)
        if (alive[j]) {
          r.first_pos[v][j] = p;
          p += o->msg_start[j + 1] - o->msg_start[j];
        }
      next = p;
    }
  }
  r.alive_end = alive;
  r.n_ver = v + 1;
  return r;
}

// The walk of a history down the tree: the message node of each matched
// message, the repos node (if any) after each matched boundary.
struct Walk {
  std::vector<Node *> msg;     // matched message nodes, in order
  std::vector<Node *> repos;   // [m]: repos node after message m (matched), else null
  Node *last = nullptr;        // deepest matched node
};

Walk walk(Node *root, const akv_oplog *o, const int32_t *tok, const std::vector<OpSet> &ops) {
  Walk w;
  w.repos.assign(o->n_msgs, nullptr);
  Node *cur = root;
  for (int m = 0; m < o->n_msgs; ++m) {
    const int64_t a = o->msg_start[m], len = o->msg_start[m + 1] - a;
    Node *mn = find_msg(cur, tok + a, len);
    if (!mn) break;
    w.msg.push_back(mn);
    cur = mn;
    if (!ops[m].empty()) {
      Node *on = find_ops(cur, ops[m]);
      if (!on) break;
      if (on->repos) w.repos[m] = on;
      cur = on;
    }
  }
  w.last = cur;
  return w;
}

}  // namespace

namespace {

// A unit's tokens as they sit in one history: its first logical token and
// the position of that token (positions inside a message are consecutive).
struct Placed {
  Unit *u;
  int64_t first_logical, first_pos;
};

struct Running {
  std::vector<Placed> active;   // newest copy of each active message, logical order (pinned)
  std::vector<Placed> written;  // units its insert gave new slots (to be filled by the caller)
  std::vector<int32_t> tail;    // slots held for decode appends
};

// Free slots of a pool as disjoint ranges [first, first + count), by first.
class FreeSlots {
 public:
  void reset(int64_t n) {
    r_.clear();
    n_ = 0;
    if (n > 0) add(0, n);
  }
  int64_t size() const { return n_; }
  // the lowest n free slots
  void take(int64_t n, std::vector<int32_t> *out) {
    while (n > 0) {
      auto it = r_.begin();
      const int64_t k = std::min<int64_t>(n, it->second);
      for (int64_t i = 0; i < k; ++i) out->push_back((int32_t)(it->first + i));
      const int64_t first = it->first + k, left = it->second - k;
      r_.erase(it);
      if (left) r_.emplace(first, left);
      n -= k;
      n_ -= k;
    }
  }
  void give(const std::vector<int32_t> &slots) {
    std::vector<int32_t> s(slots);
    std::sort(s.begin(), s.end());
    for (size_t i = 0; i < s.size();) {
      size_t j = i + 1;
      while (j < s.size() && s[j] == s[j - 1] + 1) ++j;
      add(s[i], (int64_t)(j - i));
      i = j;
    }
  }

 private:
  void add(int64_t first, int64_t count) {
    n_ += count;
    auto next = r_.lower_bound(first);
    if (next != r_.end() && next->first == first + count) {  // join the range after
      count += next->second;
      next = r_.erase(next);
    }
    if (next != r_.begin()) {
      auto prev = std::prev(next);
      if (prev->first + prev->second == first) {  // join the range before
        prev->second += count;
        return;
      }
    }
    r_.emplace(first, count);
  }
  std::map<int64_t, int64_t> r_;
  int64_t n_ = 0;
};

}  // namespace

struct akv_tree {
  Node root;
  uint64_t tick = 0;
  uint64_t units = 0;  // storage units created
  int64_t n_nodes = 1;
  int64_t pool = 0;    // slots of the managed KV pool (0: no pool)
  FreeSlots free;
  // running requests: what each one pins, was given and holds
  std::map<int64_t, Running> running;
};

namespace {

akv_status check_history(const akv_oplog *o, const int32_t *tok) {
  if (akv_status st = validate_oplog(o, -1, 0)) return st;
  if (o->msg_start[o->n_msgs] > 0 && !tok) return report_error(AKV_ERR_INVALID, "token_ids is NULL");
  return AKV_OK;
}

// Copies of message j (its node) resident for a history: the node's own KV
// (version ver_of[j]) and the re-rotated copies at the matched repos nodes
// after it (version = the version that repos opened).  Returns the version
// indices, in order of the history.
void copies_of(const Walk &w, const Replay &r, int j, std::vector<std::pair<int, Unit *>> *out) {
  out->clear();
  Node *mn = w.msg[j];
  out->push_back({r.ver_of[j], &mn->own});
  for (size_t m = j; m < w.repos.size(); ++m) {
    if (!w.repos[m]) continue;
    auto it = w.repos[m]->ver.find(mn);  // the repos after message m opened version ver_of[m] + 1
    if (it != w.repos[m]->ver.end()) out->push_back({r.ver_of[m] + 1, &it->second});
  }
}

// Free unpinned resident units (not on the path of an insert in progress)
// until `tokens` tokens are freed or none is left: dropped units first, then
// the rest, least recently used first within each class, then by creation.
// Nodes stay as empty placeholders; a pool tree gets the units' slots back.
int64_t evict_units(akv_tree *t, int64_t tokens) {
  std::vector<Unit *> cand;
  std::vector<Node *> stack{&t->root};
  while (!stack.empty()) {
    Node *nd = stack.back();
    stack.pop_back();
    if (nd->kind == Node::kMsg && nd->own.resident && nd->own.pins == 0 && !nd->own.busy)
      cand.push_back(&nd->own);
    for (auto &kv : nd->ver)
      if (kv.second.resident && kv.second.pins == 0 && !kv.second.busy) cand.push_back(&kv.second);
    for (auto &c : nd->children) stack.push_back(c.get());
  }
  std::sort(cand.begin(), cand.end(), [](const Unit *a, const Unit *b) {
    if (a->dropped != b->dropped) return a->dropped;
    if (a->last_use != b->last_use) return a->last_use < b->last_use;
    return a->seq < b->seq;
  });
  int64_t freed = 0;
  for (Unit *u : cand) {
    if (freed >= tokens) break;
    u->resident = false;  // the node stays as an empty placeholder
    freed += u->tokens;
    if (t->pool) {
      t->free.give(u->slots);
      u->slots.clear();
    }
  }
  return freed;
}

// Copy a list of placed units' slots, logical indices and positions out.
akv_status list_out(const std::vector<Placed> &list, int32_t *slots, int32_t *logical,
                    int32_t *pos, int64_t cap, int64_t *n) {
  int64_t total = 0;
  for (const Placed &p : list) total += p.u->tokens;
  *n = total;
  if (!slots && !logical && !pos) return AKV_OK;  // size query
  if (cap < total)
    return report_error(AKV_ERR_INVALID, "capacity %lld < %lld entries", (long long)cap,
                        (long long)total);
  int64_t k = 0;
  for (const Placed &p : list)
    for (int64_t i = 0; i < p.u->tokens; ++i, ++k) {
      if (slots) slots[k] = p.u->slots.empty() ? -1 : p.u->slots[i];
      if (logical) logical[k] = (int32_t)(p.first_logical + i);
      if (pos) pos[k] = (int32_t)(p.first_pos + i);
    }
  return AKV_OK;
}

}  // namespace

extern "C" {

akv_status akv_tree_create(akv_tree **out) {
  if (!out) return report_error(AKV_ERR_INVALID, "out is NULL");
  *out = new (std::nothrow) akv_tree;
  if (!*out) return report_error(AKV_ERR_INVALID, "host allocation failed");
  return AKV_OK;
}

akv_status akv_tree_create_pool(int64_t n_slots, akv_tree **out) {
  if (!out) return report_error(AKV_ERR_INVALID, "out is NULL");
  if (n_slots <= 0 || n_slots > INT32_MAX)
    return report_error(AKV_ERR_INVALID, "pool slots must be in 1..2^31-1");
  if (akv_status st = akv_tree_create(out)) return st;
  (*out)->pool = n_slots;
  (*out)->free.reset(n_slots);
  return AKV_OK;
}

void akv_tree_destroy(akv_tree *t) { delete t; }

akv_status akv_tree_match(const akv_tree *t, const akv_oplog *ops, const int32_t *token_ids,
                          akv_tree_match_result *res) {
  if (akv_status f = fault_point("akv_tree_match")) return f;
  if (!t || !res) return report_error(AKV_ERR_INVALID, "NULL argument");
  if (akv_status st = check_history(ops, token_ids)) return st;
  const std::vector<OpSet> os = op_sets(ops);
  const Replay r = replay(ops, os);
  const Walk w = walk(const_cast<Node *>(&t->root), ops, token_ids, os);
  const int n = ops->n_msgs, k = (int)w.msg.size();
  *res = akv_tree_match_result{};
  res->matched_msgs = k;
  for (int m = k; m < n; ++m) res->prefill_tokens += ops->msg_start[m + 1] - ops->msg_start[m];
  // KV the continuation reads: a full match continues from the active cache
  // at the end (at the last version's positions); a partial one prefills the
  // unmatched messages over the messages alive when the first of them starts
  const bool full = k == n;
  const std::vector<char> &need = full ? r.alive_end : r.alive_before[k];
  const int vfin = r.n_ver - 1;
  std::vector<std::pair<int, Unit *>> cp;
  for (int j = 0; j < k; ++j) {
    if (!need[j]) continue;
    const int64_t len = ops->msg_start[j + 1] - ops->msg_start[j];
    copies_of(w, r, j, &cp);
    bool resident = false, same_pos = false;
    for (auto &c : cp)
      if (c.second->resident) {
        resident = true;
        if (r.first_pos[c.first][j] == r.first_pos[vfin][j]) same_pos = true;
      }
    if (!resident) res->restore_tokens += len;
    else if (full && !same_pos) res->rotate_tokens += len;
    else res->reuse_tokens += len;
  }
  if (res->restore_tokens) res->kind = AKV_TREE_RESTORE;
  else if (!full) res->kind = AKV_TREE_PREFILL_SUFFIX;
  else if (res->rotate_tokens) res->kind = AKV_TREE_ROTATE;
  else res->kind = AKV_TREE_REUSE;
  return AKV_OK;
}

akv_status akv_tree_insert(akv_tree *t, const akv_oplog *ops, const int32_t *token_ids,
                           int64_t request_id) {
  if (akv_status f = fault_point("akv_tree_insert")) return f;
  if (!t) return report_error(AKV_ERR_INVALID, "NULL tree");
  if (akv_status st = check_history(ops, token_ids)) return st;
  if (t->running.count(request_id))
    return report_error(AKV_ERR_INVALID, "request %lld is already running",
                        (long long)request_id);
  const std::vector<OpSet> os = op_sets(ops);
  const Replay r = replay(ops, os);
  const int n = ops->n_msgs;
  const uint64_t now = ++t->tick;
  // create the path; every message's KV and every repos copy is resident now
  std::vector<Node *> msg(n, nullptr), repos(n, nullptr);
  Node *cur = &t->root;
  for (int m = 0; m < n; ++m) {
    const int64_t a = ops->msg_start[m], len = ops->msg_start[m + 1] - a;
    Node *mn = find_msg(cur, token_ids + a, len);
    if (!mn) {
      auto nn = std::make_unique<Node>();
      nn->kind = Node::kMsg;
      nn->tokens.assign(token_ids + a, token_ids + a + len);
      nn->parent = cur;
      nn->own.tokens = len;
      nn->own.seq = ++t->units;
      mn = nn.get();
      cur->children.push_back(std::move(nn));
      ++t->n_nodes;
    }
    msg[m] = mn;
    cur = mn;
    if (!os[m].empty()) {
      Node *on = find_ops(cur, os[m]);
      if (!on) {
        auto nn = std::make_unique<Node>();
        nn->kind = Node::kOps;
        nn->drops = os[m].drops;
        nn->repos = os[m].repos;
        nn->parent = cur;
        on = nn.get();
        cur->children.push_back(std::move(nn));
        ++t->n_nodes;
      }
      if (on->repos) repos[m] = on;
      cur = on;
    }
  }
  // every unit the history makes resident, in the order they are created:
  // each message's own KV, and at each repos a copy of every message alive
  std::vector<Placed> path;
  std::vector<char> alive(n, 0);
  for (int m = 0; m < n; ++m) {
    path.push_back({&msg[m]->own, ops->msg_start[m], r.first_pos[r.ver_of[m]][m]});
    alive[m] = 1;
    for (int j : os[m].drops) alive[j] = 0;
    if (repos[m])
      for (int j = 0; j <= m; ++j)
        if (alive[j]) {
          auto ins = repos[m]->ver.emplace(msg[j], Unit{});
          Unit &c = ins.first->second;
          if (ins.second) c.seq = ++t->units;
          c.tokens = ops->msg_start[j + 1] - ops->msg_start[j];
          path.push_back({&c, ops->msg_start[j], r.first_pos[r.ver_of[m] + 1][j]});
        }
  }
  // pool: slots for the units that are not resident yet, evicting other
  // unpinned units (drop-aware order) when the free list is short
  std::vector<Placed> written;
  if (t->pool) {
    // every unit sits on the path once (one per message node, one per
    // message node and repos node)
    int64_t need = 0;
    for (Placed &p : path) {
      p.u->busy = true;
      if (!p.u->resident) need += p.u->tokens;
    }
    if (t->free.size() < need) evict_units(t, need - t->free.size());
    if (t->free.size() < need) {
      for (Placed &p : path) p.u->busy = false;
      return report_error(AKV_ERR_WORKSPACE,
                          "KV pool full: %lld slots needed, %lld free after evicting every "
                          "unpinned unit", (long long)need, (long long)t->free.size());
    }
    for (Placed &p : path) {
      p.u->busy = false;
      if (!p.u->resident) {
        t->free.take(p.u->tokens, &p.u->slots);
        written.push_back(p);
      }
    }
  }
  for (Placed &p : path) {
    p.u->resident = true;
    p.u->last_use = now;
  }
  // the request's active cache at the end: the newest copy of each message
  // still alive is pinned; the rest of its path is marked by whether this
  // (latest) user dropped it
  Running &run = t->running[request_id];
  run.written = std::move(written);
  const int vfin = r.n_ver - 1;
  for (int j = 0; j < n; ++j) {
    Unit *newest = &msg[j]->own;  // the copy at the last version holding it
    for (int m = j; m < n; ++m)
      if (repos[m]) {
        auto it = repos[m]->ver.find(msg[j]);
        if (it != repos[m]->ver.end()) newest = &it->second;
      }
    const bool act = r.alive_end[j] != 0;
    msg[j]->own.dropped = !act;
    for (int m = j; m < n; ++m)
      if (repos[m]) {
        auto it = repos[m]->ver.find(msg[j]);
        if (it != repos[m]->ver.end()) it->second.dropped = !act;
      }
    if (act) {
      ++newest->pins;
      run.active.push_back({newest, ops->msg_start[j], r.first_pos[vfin][j]});
    }
  }
  return AKV_OK;
}

akv_status akv_tree_finish(akv_tree *t, int64_t request_id) {
  if (!t) return report_error(AKV_ERR_INVALID, "NULL tree");
  auto it = t->running.find(request_id);
  if (it == t->running.end())
    return report_error(AKV_ERR_INVALID, "request %lld is not running", (long long)request_id);
  for (Placed &p : it->second.active) --p.u->pins;
  if (t->pool) t->free.give(it->second.tail);
  t->running.erase(it);
  return AKV_OK;
}

akv_status akv_tree_evict(akv_tree *t, int64_t tokens, int64_t *freed) {
  if (!t || !freed) return report_error(AKV_ERR_INVALID, "NULL argument");
  *freed = evict_units(t, tokens);
  return AKV_OK;
}

akv_status akv_tree_request_cache(const akv_tree *t, int64_t request_id, int32_t *slots,
                                  int32_t *logical, int32_t *pos, int64_t cap, int64_t *n) {
  if (!t || !n) return report_error(AKV_ERR_INVALID, "NULL argument");
  auto it = t->running.find(request_id);
  if (it == t->running.end())
    return report_error(AKV_ERR_INVALID, "request %lld is not running", (long long)request_id);
  return list_out(it->second.active, slots, logical, pos, cap, n);
}

akv_status akv_tree_request_writes(const akv_tree *t, int64_t request_id, int32_t *slots,
                                   int32_t *logical, int32_t *pos, int64_t cap, int64_t *n) {
  if (!t || !n) return report_error(AKV_ERR_INVALID, "NULL argument");
  auto it = t->running.find(request_id);
  if (it == t->running.end())
    return report_error(AKV_ERR_INVALID, "request %lld is not running", (long long)request_id);
  return list_out(it->second.written, slots, logical, pos, cap, n);
}

akv_status akv_tree_reserve(akv_tree *t, int64_t request_id, int64_t n, int32_t *slots) {
  if (!t || (n > 0 && !slots) || n < 0) return report_error(AKV_ERR_INVALID, "bad argument");
  if (!t->pool) return report_error(AKV_ERR_INVALID, "the tree manages no pool");
  auto it = t->running.find(request_id);
  if (it == t->running.end())
    return report_error(AKV_ERR_INVALID, "request %lld is not running", (long long)request_id);
  if (t->free.size() < n) evict_units(t, n - t->free.size());
  if (t->free.size() < n)
    return report_error(AKV_ERR_WORKSPACE, "KV pool full: %lld slots asked, %lld free",
                        (long long)n, (long long)t->free.size());
  std::vector<int32_t> got;
  t->free.take(n, &got);
  std::copy(got.begin(), got.end(), slots);
  it->second.tail.insert(it->second.tail.end(), got.begin(), got.end());
  return AKV_OK;
}

akv_status akv_tree_pool_info(const akv_tree *t, int64_t *pool_slots, int64_t *free_slots) {
  if (!t || !pool_slots || !free_slots) return report_error(AKV_ERR_INVALID, "NULL argument");
  *pool_slots = t->pool;
  *free_slots = t->pool ? t->free.size() : 0;
  return AKV_OK;
}

akv_status akv_tree_stats(const akv_tree *t, akv_tree_stats_t *st) {
  if (!t || !st) return report_error(AKV_ERR_INVALID, "NULL argument");
  *st = akv_tree_stats_t{};
  st->nodes = t->n_nodes;
  st->running = (int64_t)t->running.size();
  std::vector<const Node *> stack{&t->root};
  while (!stack.empty()) {
    const Node *nd = stack.back();
    stack.pop_back();
    if (nd->kind == Node::kMsg) {
      if (nd->own.resident) st->resident_tokens += nd->own.tokens;
      if (nd->own.pins) st->pinned_tokens += nd->own.tokens;
    }
    for (auto &kv : nd->ver) {
      if (kv.second.resident) st->resident_tokens += kv.second.tokens;
      if (kv.second.pins) st->pinned_tokens += kv.second.tokens;
    }
    for (auto &c : nd->children) stack.push_back(c.get());
  }
  return AKV_OK;
}

}  // extern "C"
