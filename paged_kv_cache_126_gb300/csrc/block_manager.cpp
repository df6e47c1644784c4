// Host block manager: free-list paging with reference counts, zero-copy fork,
// copy-on-write of the tail frame, and prefix caching of filled blocks.
//
// Behaviour follows "PagedAttention: Virtual Memory Guide for LLM Inference"
// ("The Mathematics of Block Translation"; "Key Architectural Mechanics" 1-2;
// "Reference Implementation: Block Table & Paged Cache Manager"; "2. Native
// Synergy with RadixAttention and Prompt Caching": filled blocks are immutable, so
// an identical token prefix maps onto the frames that already hold it), "Solving
// the LLM Memory Wall" (BlockManager.allocate: a prompt's frames are granted
// all-or-nothing) and the worked trace of "PagedAttention, simply explained".
//
// Data structures: the free list is a doubly linked list over frame ids (pop at
// the front, push at the back, and removal of a freed cached frame that a new
// prompt reuses, all O(1)); sequences live in a hash map id -> {frame table,
// length, and for prompts admitted with token ids the tokens and the block nodes}.
// Filled blocks with known tokens form a trie: node = (parent node, the block's B
// token ids) -> frame, node ids never reused.  A freed cached frame keeps its node
// until the free list hands it out again.  A decode step is made all-or-nothing
// with an undo log replayed in reverse on failure, which restores the free-list
// order, evicted nodes and registrations exactly.
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <new>
#include <unordered_map>
#include <vector>

#include "pa.h"

namespace {

class FreeList {
 public:
  void reset(int32_t n) {
    prev_.assign(n, -1);
    next_.assign(n, -1);
    in_.assign(n, 0);
    head_ = tail_ = -1;
    count_ = 0;
  }
  int32_t size() const { return count_; }
  bool contains(int32_t f) const { return in_[f] != 0; }
  int32_t front() const { return head_; }
  int32_t next(int32_t f) const { return next_[f]; }
  int32_t pop_front() {
    const int32_t f = head_;
    remove(f);
    return f;
  }
  void push_back(int32_t f) {
    prev_[f] = tail_;
    next_[f] = -1;
    if (tail_ >= 0) next_[tail_] = f; else head_ = f;
    tail_ = f;
    in_[f] = 1;
    ++count_;
  }
  void push_front(int32_t f) {
    next_[f] = head_;
    prev_[f] = -1;
    if (head_ >= 0) prev_[head_] = f; else tail_ = f;
    head_ = f;
    in_[f] = 1;
    ++count_;
  }
  void remove(int32_t f) {
    const int32_t p = prev_[f], n = next_[f];
    if (p >= 0) next_[p] = n; else head_ = n;
    if (n >= 0) prev_[n] = p; else tail_ = p;
    in_[f] = 0;
    --count_;
  }

 private:
  std::vector<int32_t> prev_, next_;
  std::vector<uint8_t> in_;
  int32_t head_ = -1, tail_ = -1, count_ = 0;
};

constexpr int64_t kUnknownToken = INT64_MIN;

// A filled block's identity: the node of the block before it (0 at the start of a
// sequence) and its token ids.
struct BlockKey {
  int64_t parent;
  std::vector<int32_t> tokens;
  bool operator==(const BlockKey& o) const { return parent == o.parent && tokens == o.tokens; }
};
struct BlockKeyHash {
  size_t operator()(const BlockKey& k) const {
    uint64_t h = 1469598103934665603ull ^ static_cast<uint64_t>(k.parent);
    h *= 1099511628211ull;
    for (int32_t t : k.tokens) {
      h ^= static_cast<uint32_t>(t);
      h *= 1099511628211ull;
    }
    return static_cast<size_t>(h);
  }
};
struct Node {
  int32_t frame;
  BlockKey key;
};

struct Seq {
  std::vector<int32_t> frames;
  int32_t len = 0;
  bool tracked = false;         // admitted with token ids: tokens and nodes are kept
  std::vector<int64_t> tokens;  // kUnknownToken where an append carried no id
  std::vector<int64_t> nodes;   // node standing for each block's content, 0: none
};

// What one append did, so a failed step can be rolled back.
struct Undo {
  enum Kind : uint8_t { kInPlace, kNewFrame, kCopyOnWrite } kind;
  int64_t seq;
  int32_t taken;        // frame popped from the free list (kNewFrame, kCopyOnWrite)
  int32_t shared;       // frame replaced in the table (kCopyOnWrite)
  int64_t evicted = 0;  // node evicted from `taken` when it left the free list
  Node evicted_node{};
  int64_t registered = 0;  // node created because this append filled a block
  bool mapped = false;     // the filled block was given a node (new or existing)
};

}  // namespace

struct pa_bm {
  int32_t num_blocks = 0;
  int32_t block_size = 0;
  FreeList free_list;
  std::vector<int32_t> refs;
  using SeqMap = std::unordered_map<int64_t, Seq>;
  SeqMap seqs;
  // Map nodes of freed sequences, kept with their vectors' capacity and reused by forks:
  // a beam-search step that forks and frees as many sequences as it keeps then
  // allocates nothing.
  static constexpr size_t kSpareMax = 4096;
  std::vector<SeqMap::node_type> spare;
  // prefix cache
  std::unordered_map<BlockKey, int64_t, BlockKeyHash> node_of_key;
  std::unordered_map<int64_t, Node> nodes;
  std::vector<int64_t> frame_node;  // node registered on each frame, 0: none
  int64_t next_node = 1;

  int32_t slot_of(const Seq& s, int32_t pos) const {
    return s.frames[pos / block_size] * block_size + pos % block_size;
  }

  // slots of positions [from, to) of s into out[0 .. to-from), frame by frame (no
  // division per token: a prompt's slots are most of its admission's host time)
  void slots_of(const Seq& s, int32_t from, int32_t to, int32_t* out) const {
    int32_t pos = from;
    while (pos < to) {
      const int32_t b = pos / block_size;
      const int32_t off = pos - b * block_size;
      const int32_t end = std::min(to, (b + 1) * block_size);
      const int32_t base = s.frames[b] * block_size;
      for (int32_t o = off; pos < end; ++pos, ++o) *out++ = base + o;
    }
  }

  // Pops the front frame; a frame still holding a cached block loses its node.
  int32_t take_frame(Undo* u) {
    const int32_t f = free_list.pop_front();
    refs[f] = 1;
    const int64_t node = frame_node[f];
    if (node) {
      auto it = nodes.find(node);
      if (u) {
        u->evicted = node;
        u->evicted_node = it->second;
      }
      node_of_key.erase(it->second.key);
      nodes.erase(it);
      frame_node[f] = 0;
    }
    return f;
  }

  // Fork of a live parent into a child id known not to be live: the child shares every
  // frame (each gains a reference) and inherits the length.  The child is inserted before
  // any reference count moves, so a failed allocation leaves the manager as it was.
  void fork_checked(const Seq& parent, int64_t child_id) {
    SeqMap::iterator at;
    if (!spare.empty()) {
      // a recycled node: copying into vectors that keep their capacity allocates nothing
      SeqMap::node_type nh = std::move(spare.back());
      spare.pop_back();
      nh.key() = child_id;
      Seq& c = nh.mapped();
      c.frames.assign(parent.frames.begin(), parent.frames.end());
      c.len = parent.len;
      c.tracked = parent.tracked;
      c.tokens.assign(parent.tokens.begin(), parent.tokens.end());
      c.nodes.assign(parent.nodes.begin(), parent.nodes.end());
      at = seqs.insert(std::move(nh)).position;
    } else {
      Seq child = parent;  // copy of the table and the length (the insert may rehash: copy first)
      at = seqs.emplace(child_id, std::move(child)).first;
    }
    for (int32_t f : at->second.frames) refs[f] += 1;
  }

  // Removes a live sequence's map entry, keeping its node for a later fork.
  void erase_seq(SeqMap::iterator it) {
    if (spare.size() >= kSpareMax) {
      seqs.erase(it);
      return;
    }
    SeqMap::node_type nh = seqs.extract(it);
    try {
      spare.push_back(std::move(nh));
    } catch (...) {  // no room to keep it: the node handle frees it
    }
  }

  void drop_ref(int32_t f) {
    if (refs[f] <= 0) return;  // already free: releasing again does nothing
    if (--refs[f] == 0) free_list.push_back(f);
  }

  // Block `block` of s has just been filled; give it a node if its tokens are known
  // and the block before it has one.  Returns the node created (0 if none was).
  int64_t register_block(Seq& s, int32_t block, bool* mapped) {
    *mapped = false;
    const int64_t parent = block == 0 ? 0 : s.nodes[block - 1];
    if (block > 0 && parent == 0) return 0;
    BlockKey key{parent, std::vector<int32_t>(block_size)};
    for (int32_t j = 0; j < block_size; ++j) {
      const int64_t t = s.tokens[static_cast<size_t>(block) * block_size + j];
      if (t == kUnknownToken) return 0;
      key.tokens[j] = static_cast<int32_t>(t);
    }
    *mapped = true;
    auto it = node_of_key.find(key);
    if (it != node_of_key.end()) {  // the same content is registered already
      s.nodes[block] = it->second;
      return 0;
    }
    const int64_t node = next_node++;
    const int32_t frame = s.frames[block];
    nodes.emplace(node, Node{frame, key});
    node_of_key.emplace(std::move(key), node);
    frame_node[frame] = node;
    s.nodes[block] = node;
    return node;
  }

  void unregister(int64_t node) {
    auto it = nodes.find(node);
    frame_node[it->second.frame] = 0;
    node_of_key.erase(it->second.key);
    nodes.erase(it);
  }

  // One append (token id or kUnknownToken); on success fills *slot and the copy pair
  // and records an undo entry.
  int append_one(int64_t id, int64_t token, int32_t* slot, int32_t* src, int32_t* dst, std::vector<Undo>* log) {
    auto it = seqs.find(id);
    if (it == seqs.end()) return PA_ERR_UNKNOWN_SEQ;
    Seq& s = it->second;
    const int32_t t = s.len;
    *src = -1;
    *dst = -1;
    Undo u{Undo::kInPlace, id, -1, -1};
    if (t % block_size == 0) {  // boundary: the current frame is full (or none yet)
      if (free_list.size() == 0) return PA_ERR_OUT_OF_BLOCKS;
      u.kind = Undo::kNewFrame;
      u.taken = take_frame(&u);
      s.frames.push_back(u.taken);
      if (s.tracked) s.nodes.push_back(0);
    } else {
      const int32_t tail = s.frames.back();
      if (refs[tail] > 1) {  // shared tail: move this writer onto a private copy
        if (free_list.size() == 0) return PA_ERR_OUT_OF_BLOCKS;
        u.kind = Undo::kCopyOnWrite;
        u.taken = take_frame(&u);
        u.shared = tail;
        drop_ref(tail);
        s.frames.back() = u.taken;
        *src = tail;
        *dst = u.taken;
      }
    }
    s.len = t + 1;
    *slot = slot_of(s, t);
    if (s.tracked) {
      s.tokens.push_back(token);
      if ((t + 1) % block_size == 0) u.registered = register_block(s, t / block_size, &u.mapped);
    }
    if (log) log->push_back(std::move(u));
    return PA_OK;
  }

  void undo(const Undo& u) {
    Seq& s = seqs[u.seq];
    s.len -= 1;
    if (s.tracked) {
      if (u.registered) unregister(u.registered);
      if (u.mapped) s.nodes[s.len / block_size] = 0;
      s.tokens.pop_back();
    }
    switch (u.kind) {
      case Undo::kInPlace:
        break;
      case Undo::kNewFrame:
        s.frames.pop_back();
        if (s.tracked) s.nodes.pop_back();
        refs[u.taken] = 0;
        free_list.push_front(u.taken);
        break;
      case Undo::kCopyOnWrite:
        s.frames.back() = u.shared;
        refs[u.shared] += 1;  // copy-on-write only runs on a frame with more than one reference
        refs[u.taken] = 0;
        free_list.push_front(u.taken);
        break;
    }
    if (u.evicted) {  // the frame goes back to holding its cached block
      nodes.emplace(u.evicted, u.evicted_node);
      node_of_key.emplace(u.evicted_node.key, u.evicted);
      frame_node[u.evicted_node.frame] = u.evicted;
    }
  }

  // Appends a run of tokens (one sequence or several), all-or-nothing.
  int run_appends(const int64_t* ids, int64_t single_id, const int32_t* tokens, int32_t n, int32_t* slots_out,
                  int32_t* copies_out, int32_t* n_copies_out) {
    std::vector<Undo> log;
    log.reserve(n);
    const int64_t saved_next = next_node;
    int32_t n_copies = 0;
    for (int32_t i = 0; i < n; ++i) {
      int32_t src, dst;
      const int64_t id = ids ? ids[i] : single_id;
      const int64_t tok = tokens ? static_cast<int64_t>(tokens[i]) : kUnknownToken;
      int rc = append_one(id, tok, &slots_out[i], &src, &dst, &log);
      if (rc != PA_OK) {
        for (auto u = log.rbegin(); u != log.rend(); ++u) undo(*u);
        next_node = saved_next;
        return rc;
      }
      if (src >= 0) {
        if (copies_out) {
          copies_out[2 * n_copies] = src;
          copies_out[2 * n_copies + 1] = dst;
        }
        ++n_copies;
      }
    }
    if (n_copies_out) *n_copies_out = n_copies;
    return PA_OK;
  }
};

// Every entry point runs inside guarded(): no C++ exception crosses the C ABI.  A failed
// host allocation returns PA_ERR_HOST_MEMORY (the manager's state may then be partly
// changed: operations are all-or-nothing for lack of frames, not for lack of host memory).
template <typename F>
int guarded(F&& f) noexcept {
  try {
    return f();
  } catch (const std::bad_alloc&) {
    return PA_ERR_HOST_MEMORY;
  } catch (...) {
    return PA_ERR_INVALID;
  }
}

extern "C" {

int pa_bm_create(int32_t num_blocks, int32_t block_size, const int32_t* free_order, pa_bm** bm_out) {
  return guarded([&]() -> int {
    if (!bm_out || num_blocks <= 0 || block_size <= 0) return PA_ERR_INVALID;
    if (static_cast<int64_t>(num_blocks) * block_size > INT32_MAX) return PA_ERR_INVALID;
    pa_bm* bm = new (std::nothrow) pa_bm();
    if (!bm) return PA_ERR_INVALID;
    bm->num_blocks = num_blocks;
    bm->block_size = block_size;
    bm->refs.assign(num_blocks, 0);
    bm->frame_node.assign(num_blocks, 0);
    // at most one registered block per frame: the prefix-cache maps never rehash
    bm->node_of_key.reserve(static_cast<size_t>(num_blocks));
    bm->nodes.reserve(static_cast<size_t>(num_blocks));
    bm->spare.reserve(pa_bm::kSpareMax);
    bm->free_list.reset(num_blocks);
    if (free_order) {
      std::vector<uint8_t> seen(num_blocks, 0);
      for (int32_t i = 0; i < num_blocks; ++i) {
        int32_t f = free_order[i];
        if (f < 0 || f >= num_blocks || seen[f]) {
          delete bm;
          return PA_ERR_INVALID;
        }
        seen[f] = 1;
        bm->free_list.push_back(f);
      }
    } else {
      for (int32_t i = 0; i < num_blocks; ++i) bm->free_list.push_back(i);
    }
    *bm_out = bm;
    return PA_OK;
  });
}

void pa_bm_destroy(pa_bm* bm) { delete bm; }

int pa_bm_add_seq(pa_bm* bm, int64_t seq_id, int32_t num_tokens, int32_t* slots_out) {
  return guarded([&]() -> int {
    if (!bm || num_tokens < 0) return PA_ERR_INVALID;
    if (bm->seqs.count(seq_id)) return PA_ERR_SEQ_EXISTS;
    const int32_t need = num_tokens / bm->block_size + (num_tokens % bm->block_size != 0);
    if (need > bm->free_list.size()) return PA_ERR_OUT_OF_BLOCKS;
    Seq s;
    s.frames.reserve(need + 1);
    for (int32_t j = 0; j < need; ++j) s.frames.push_back(bm->take_frame(nullptr));
    s.len = num_tokens;
    if (slots_out)
      bm->slots_of(s, 0, num_tokens, slots_out);
    bm->seqs.emplace(seq_id, std::move(s));
    return PA_OK;
  });
}

int pa_bm_append(pa_bm* bm, int64_t seq_id, int32_t* slot_out, int32_t* cow_src, int32_t* cow_dst) {
  return guarded([&]() -> int {
    if (!bm || !slot_out) return PA_ERR_INVALID;
    int32_t src, dst;
    int rc = bm->append_one(seq_id, kUnknownToken, slot_out, &src, &dst, nullptr);
    if (rc != PA_OK) return rc;
    if (cow_src) *cow_src = src;
    if (cow_dst) *cow_dst = dst;
    return PA_OK;
  });
}

int pa_bm_step(pa_bm* bm, const int64_t* seq_ids, int32_t n, int32_t* slots_out,
               int32_t* copies_out, int32_t* n_copies_out) {
  return guarded([&]() -> int {
    if (!bm || n < 0 || (n > 0 && (!seq_ids || !slots_out))) return PA_ERR_INVALID;
    return bm->run_appends(seq_ids, 0, nullptr, n, slots_out, copies_out, n_copies_out);
  });
}

int pa_bm_step_tokens(pa_bm* bm, const int64_t* seq_ids, const int32_t* tokens, int32_t n, int32_t* slots_out,
                      int32_t* copies_out, int32_t* n_copies_out) {
  return guarded([&]() -> int {
    if (!bm || n < 0 || (n > 0 && (!seq_ids || !tokens || !slots_out))) return PA_ERR_INVALID;
    return bm->run_appends(seq_ids, 0, tokens, n, slots_out, copies_out, n_copies_out);
  });
}

int pa_bm_extend(pa_bm* bm, int64_t seq_id, int32_t num_tokens, int32_t* slots_out, int32_t* copies_out,
                 int32_t* n_copies_out) {
  return guarded([&]() -> int {
    if (!bm || num_tokens < 0 || (num_tokens > 0 && !slots_out)) return PA_ERR_INVALID;
    if (!bm->seqs.count(seq_id)) return PA_ERR_UNKNOWN_SEQ;
    return bm->run_appends(nullptr, seq_id, nullptr, num_tokens, slots_out, copies_out, n_copies_out);
  });
}

int pa_bm_extend_tokens(pa_bm* bm, int64_t seq_id, const int32_t* tokens, int32_t num_tokens, int32_t* slots_out,
                        int32_t* copies_out, int32_t* n_copies_out) {
  return guarded([&]() -> int {
    if (!bm || num_tokens < 0 || (num_tokens > 0 && (!slots_out || !tokens))) return PA_ERR_INVALID;
    if (!bm->seqs.count(seq_id)) return PA_ERR_UNKNOWN_SEQ;
    return bm->run_appends(nullptr, seq_id, tokens, num_tokens, slots_out, copies_out, n_copies_out);
  });
}

int pa_bm_add_seq_cached(pa_bm* bm, int64_t seq_id, const int32_t* tokens, int32_t num_tokens,
                         int32_t* slots_out, int32_t* n_cached_out) {
  return guarded([&]() -> int {
    if (!bm || num_tokens < 0 || (num_tokens > 0 && (!tokens || !slots_out))) return PA_ERR_INVALID;
    if (bm->seqs.count(seq_id)) return PA_ERR_SEQ_EXISTS;
    const int32_t B = bm->block_size, L = num_tokens;
    // leading filled blocks already cached; the last token is never among them
    std::vector<int64_t> hit_nodes;
    std::vector<int32_t> hit_frames;
    int64_t parent = 0;
    BlockKey key{0, std::vector<int32_t>(B)};
    while (static_cast<int64_t>(hit_nodes.size() + 1) * B <= static_cast<int64_t>(L) - 1) {
      const size_t i = hit_nodes.size();
      key.parent = parent;
      std::memcpy(key.tokens.data(), tokens + i * B, sizeof(int32_t) * B);
      auto it = bm->node_of_key.find(key);
      if (it == bm->node_of_key.end()) break;
      hit_nodes.push_back(it->second);
      hit_frames.push_back(bm->nodes.find(it->second)->second.frame);
      parent = it->second;
    }
    const int32_t n_hits = static_cast<int32_t>(hit_nodes.size());
    const int32_t n_blocks = L / B + (L % B != 0);
    int32_t available = bm->free_list.size();
    for (int32_t f : hit_frames)
      if (bm->refs[f] == 0) --available;
    if (n_blocks - n_hits > available) return PA_ERR_OUT_OF_BLOCKS;
    for (int32_t f : hit_frames) {  // reuse: a freed cached frame leaves the free list
      if (bm->refs[f] == 0) bm->free_list.remove(f);
      bm->refs[f] += 1;
    }
    Seq s;
    s.tracked = true;
    s.len = L;
    s.frames = hit_frames;
    s.nodes = hit_nodes;
    s.tokens.assign(tokens, tokens + L);
    s.frames.reserve(n_blocks + 1);
    for (int32_t i = n_hits; i < n_blocks; ++i) {
      s.frames.push_back(bm->take_frame(nullptr));
      s.nodes.push_back(0);
      bool mapped;
      if (static_cast<int64_t>(i + 1) * B <= L) bm->register_block(s, i, &mapped);
    }
    const int32_t n_cached = n_hits * B;
    bm->slots_of(s, n_cached, L, slots_out);
    if (n_cached_out) *n_cached_out = n_cached;
    bm->seqs.emplace(seq_id, std::move(s));
    return PA_OK;
  });
}

int pa_bm_cached_frames(const pa_bm* bm, int32_t* out, int32_t cap, int32_t* n_cached_out) {
  return guarded([&]() -> int {
    if (!bm || cap < 0 || (cap > 0 && !out)) return PA_ERR_INVALID;
    if (out && cap < bm->num_blocks) return PA_ERR_CAPACITY;
    int32_t n = 0;
    for (int32_t f = 0; f < bm->num_blocks; ++f) {
      const int32_t c = bm->frame_node[f] != 0;
      if (out) out[f] = c;
      n += c;
    }
    if (n_cached_out) *n_cached_out = n;
    return PA_OK;
  });
}

int pa_bm_fork(pa_bm* bm, int64_t parent_id, int64_t child_id) {
  return guarded([&]() -> int {
    if (!bm) return PA_ERR_INVALID;
    auto p = bm->seqs.find(parent_id);
    if (p == bm->seqs.end()) return PA_ERR_UNKNOWN_SEQ;
    if (bm->seqs.count(child_id)) return PA_ERR_SEQ_EXISTS;
    bm->fork_checked(p->second, child_id);
    return PA_OK;
  });
}

int pa_bm_free(pa_bm* bm, int64_t seq_id) {
  return guarded([&]() -> int {
    if (!bm) return PA_ERR_INVALID;
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return PA_WARN_DOUBLE_FREE;
    for (int32_t f : it->second.frames) bm->drop_ref(f);
    bm->erase_seq(it);
    return PA_OK;
  });
}

int pa_bm_fork_many(pa_bm* bm, const int64_t* parent_ids, const int64_t* child_ids, int32_t n) {
  return guarded([&]() -> int {
    if (!bm || n < 0 || (n > 0 && (!parent_ids || !child_ids))) return PA_ERR_INVALID;
    // all-or-nothing: check the whole batch in order (a child forked earlier in the batch may
    // be a later parent) before changing anything.  born = (child id, position) sorted, so
    // "x is a child of an earlier fork" is one binary search: the first position of x < i.
    std::vector<std::pair<int64_t, int32_t>> born(static_cast<size_t>(n));
    for (int32_t i = 0; i < n; ++i) born[i] = {child_ids[i], i};
    std::sort(born.begin(), born.end());
    auto born_before = [&](int64_t x, int32_t i) {
      const auto it = std::lower_bound(born.begin(), born.end(), std::make_pair(x, INT32_MIN));
      return it != born.end() && it->first == x && it->second < i;
    };
    for (int32_t i = 0; i < n; ++i) {
      if (!bm->seqs.count(parent_ids[i]) && !born_before(parent_ids[i], i)) return PA_ERR_UNKNOWN_SEQ;
      if (bm->seqs.count(child_ids[i]) || born_before(child_ids[i], i)) return PA_ERR_SEQ_EXISTS;
    }
    for (int32_t i = 0; i < n; ++i) bm->fork_checked(bm->seqs.find(parent_ids[i])->second, child_ids[i]);
    return PA_OK;
  });
}

int pa_bm_free_many(pa_bm* bm, const int64_t* seq_ids, int32_t n) {
  return guarded([&]() -> int {
    if (!bm || n < 0 || (n > 0 && !seq_ids)) return PA_ERR_INVALID;
    int rc = PA_OK;
    for (int32_t i = 0; i < n; ++i)
      if (pa_bm_free(bm, seq_ids[i]) == PA_WARN_DOUBLE_FREE) rc = PA_WARN_DOUBLE_FREE;
    return rc;
  });
}

int pa_bm_block_tables(const pa_bm* bm, const int64_t* seq_ids, int32_t n, int32_t max_blocks,
                       int32_t* tables_out, int32_t* lens_out) {
  return guarded([&]() -> int {
    if (!bm || n < 0 || max_blocks < 0 || (n > 0 && (!seq_ids || (!tables_out && max_blocks > 0))))
      return PA_ERR_INVALID;
    for (int32_t i = 0; i < n; ++i) {
      auto it = bm->seqs.find(seq_ids[i]);
      if (it == bm->seqs.end()) return PA_ERR_UNKNOWN_SEQ;
      if (static_cast<int32_t>(it->second.frames.size()) > max_blocks) return PA_ERR_CAPACITY;
    }
    for (int32_t i = 0; i < n; ++i) {
      const Seq& s = bm->seqs.find(seq_ids[i])->second;
      int32_t* row = tables_out + static_cast<int64_t>(i) * max_blocks;
      const int32_t nf = static_cast<int32_t>(s.frames.size());
      if (nf) std::memcpy(row, s.frames.data(), sizeof(int32_t) * nf);
      for (int32_t j = nf; j < max_blocks; ++j) row[j] = -1;
      if (lens_out) lens_out[i] = s.len;
    }
    return PA_OK;
  });
}

int pa_bm_seq_info(const pa_bm* bm, int64_t seq_id, int32_t* len_out, int32_t* n_blocks_out) {
  return guarded([&]() -> int {
    if (!bm) return PA_ERR_INVALID;
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return PA_ERR_UNKNOWN_SEQ;
    if (len_out) *len_out = it->second.len;
    if (n_blocks_out) *n_blocks_out = static_cast<int32_t>(it->second.frames.size());
    return PA_OK;
  });
}

int pa_bm_table(const pa_bm* bm, int64_t seq_id, int32_t* out, int32_t cap, int32_t* n_out) {
  return guarded([&]() -> int {
    if (!bm || cap < 0 || (cap > 0 && !out)) return PA_ERR_INVALID;
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return PA_ERR_UNKNOWN_SEQ;
    const auto& fr = it->second.frames;
    if (n_out) *n_out = static_cast<int32_t>(fr.size());
    if (static_cast<int32_t>(fr.size()) > cap) return PA_ERR_CAPACITY;
    if (!fr.empty()) std::memcpy(out, fr.data(), sizeof(int32_t) * fr.size());
    return PA_OK;
  });
}

int pa_bm_slot(const pa_bm* bm, int64_t seq_id, int32_t pos, int32_t* slot_out) {
  return guarded([&]() -> int {
    if (!bm || !slot_out) return PA_ERR_INVALID;
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return PA_ERR_UNKNOWN_SEQ;
    if (pos < 0 || pos >= it->second.len) return PA_ERR_INVALID;
    *slot_out = bm->slot_of(it->second, pos);
    return PA_OK;
  });
}

int pa_bm_num_free(const pa_bm* bm, int32_t* n_out) {
  return guarded([&]() -> int {
    if (!bm || !n_out) return PA_ERR_INVALID;
    *n_out = bm->free_list.size();
    return PA_OK;
  });
}

int pa_bm_free_list(const pa_bm* bm, int32_t* out, int32_t cap, int32_t* n_out) {
  return guarded([&]() -> int {
    if (!bm || cap < 0 || (cap > 0 && !out)) return PA_ERR_INVALID;
    const int32_t n = bm->free_list.size();
    if (n_out) *n_out = n;
    if (n > cap) return PA_ERR_CAPACITY;
    int32_t i = 0;
    for (int32_t f = bm->free_list.front(); f >= 0; f = bm->free_list.next(f)) out[i++] = f;
    return PA_OK;
  });
}

int pa_bm_ref_counts(const pa_bm* bm, int32_t* out, int32_t cap) {
  return guarded([&]() -> int {
    if (!bm || !out) return PA_ERR_INVALID;
    if (cap < bm->num_blocks) return PA_ERR_CAPACITY;
    std::memcpy(out, bm->refs.data(), sizeof(int32_t) * bm->num_blocks);
    return PA_OK;
  });
}

int pa_bm_num_seqs(const pa_bm* bm, int32_t* n_out) {
  return guarded([&]() -> int {
    if (!bm || !n_out) return PA_ERR_INVALID;
    *n_out = static_cast<int32_t>(bm->seqs.size());
    return PA_OK;
  });
}

int pa_bm_export(const pa_bm* bm, int64_t* ids_out, int32_t* lens_out, int64_t* table_offsets_out,
                 int32_t* tables_out, int32_t* free_out, int32_t* refs_out, int32_t cap_seqs,
                 int64_t cap_entries, int32_t* n_seqs_out, int64_t* n_entries_out, int32_t* n_free_out) {
  return guarded([&]() -> int {
    if (!bm || cap_seqs < 0 || cap_entries < 0 || !ids_out || !lens_out || !table_offsets_out ||
        (cap_entries > 0 && !tables_out) || !free_out || !refs_out)
      return PA_ERR_INVALID;
    std::vector<int64_t> ids;
    ids.reserve(bm->seqs.size());
    int64_t entries = 0;
    for (const auto& kv : bm->seqs) {
      ids.push_back(kv.first);
      entries += static_cast<int64_t>(kv.second.frames.size());
    }
    std::sort(ids.begin(), ids.end());
    const int64_t n = static_cast<int64_t>(ids.size());
    if (n_seqs_out) *n_seqs_out = static_cast<int32_t>(n);
    if (n_entries_out) *n_entries_out = entries;
    if (n_free_out) *n_free_out = bm->free_list.size();
    if (n > cap_seqs || entries > cap_entries) return PA_ERR_CAPACITY;
    int64_t off = 0;
    for (int64_t i = 0; i < n; ++i) {
      const Seq& s = bm->seqs.find(ids[i])->second;
      ids_out[i] = ids[i];
      lens_out[i] = s.len;
      table_offsets_out[i] = off;
      if (!s.frames.empty()) std::memcpy(tables_out + off, s.frames.data(), sizeof(int32_t) * s.frames.size());
      off += static_cast<int64_t>(s.frames.size());
    }
    table_offsets_out[n] = off;
    int32_t k = 0;
    for (int32_t f = bm->free_list.front(); f >= 0; f = bm->free_list.next(f)) free_out[k++] = f;
    std::memcpy(refs_out, bm->refs.data(), sizeof(int32_t) * bm->num_blocks);
    return PA_OK;
  });
}

int pa_bm_usage(const pa_bm* bm, pa_bm_usage_t* out) {
  return guarded([&]() -> int {
    if (!bm || !out) return PA_ERR_INVALID;
    const int64_t B = bm->block_size;
    pa_bm_usage_t u{};
    u.num_seqs = static_cast<int64_t>(bm->seqs.size());
    u.frames_total = bm->num_blocks;
    std::vector<int32_t> fill(bm->num_blocks, 0);  // largest fill any sharer gives a frame
    for (const auto& kv : bm->seqs) {
      const Seq& s = kv.second;
      const int64_t nf = static_cast<int64_t>(s.frames.size());
      u.table_entries += nf;
      u.tokens_logical += s.len;
      u.max_seq_waste = std::max(u.max_seq_waste, nf * B - s.len);
      for (int64_t i = 0; i < nf; ++i) {
        const int32_t f = static_cast<int32_t>(std::min(B, std::max<int64_t>(0, s.len - i * B)));
        int32_t& slot = fill[s.frames[i]];
        slot = std::max(slot, f);
      }
    }
    for (int32_t f = 0; f < bm->num_blocks; ++f) {
      if (bm->refs[f] > 0) {
        ++u.frames_in_use;
        u.slots_filled += fill[f];
      } else if (bm->frame_node[f] != 0 && bm->free_list.contains(f)) {
        ++u.frames_cached;
      }
    }
    *out = u;
    return PA_OK;
  });
}

}  // extern "C"
