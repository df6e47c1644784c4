// Host block manager: free-list paging with reference counts, zero-copy fork and
// copy-on-write of the tail frame.
//
// Behaviour follows "PagedAttention: Virtual Memory Guide for LLM Inference"
// ("The Mathematics of Block Translation"; "Key Architectural Mechanics" 1-2;
// "Reference Implementation: Block Table & Paged Cache Manager"), "Solving the
// LLM Memory Wall" (BlockManager.allocate: a prompt's frames are granted
// all-or-nothing) and the worked trace of "PagedAttention, simply explained".
//
// Data structures: the free list is a ring buffer (pop at the front, push at the
// back, O(1)); sequences live in a hash map id -> {frame table, length}.  A decode
// step is made all-or-nothing with an undo log replayed in reverse on failure,
// which restores the free-list order exactly.
#include <cstdint>
#include <cstring>
#include <new>
#include <unordered_map>
#include <vector>

#include "pa.h"

namespace {

class FrameRing {
 public:
  void reset(int32_t capacity) {
    buf_.assign(capacity, 0);
    head_ = 0;
    count_ = 0;
  }
  int32_t size() const { return count_; }
  int32_t capacity() const { return static_cast<int32_t>(buf_.size()); }
  int32_t pop_front() {
    int32_t f = buf_[head_];
    head_ = (head_ + 1 == capacity()) ? 0 : head_ + 1;
    --count_;
    return f;
  }
  void push_back(int32_t f) {
    int32_t tail = head_ + count_;
    if (tail >= capacity()) tail -= capacity();
    buf_[tail] = f;
    ++count_;
  }
  void push_front(int32_t f) {
    head_ = (head_ == 0) ? capacity() - 1 : head_ - 1;
    buf_[head_] = f;
    ++count_;
  }
  int32_t at(int32_t i) const {  // i-th from the front
    int32_t j = head_ + i;
    if (j >= capacity()) j -= capacity();
    return buf_[j];
  }

 private:
  std::vector<int32_t> buf_;
  int32_t head_ = 0, count_ = 0;
};

struct Seq {
  std::vector<int32_t> frames;
  int32_t len = 0;
};

// What one append did, so a failed step can be rolled back.
struct Undo {
  enum Kind : uint8_t { kInPlace, kNewFrame, kCopyOnWrite } kind;
  int64_t seq;
  int32_t taken;   // frame popped from the free list (kNewFrame, kCopyOnWrite)
  int32_t shared;  // frame replaced in the table (kCopyOnWrite)
};

}  // namespace

struct pa_bm {
  int32_t num_blocks = 0;
  int32_t block_size = 0;
  FrameRing free_list;
  std::vector<int32_t> refs;
  std::unordered_map<int64_t, Seq> seqs;

  int32_t slot_of(const Seq& s, int32_t pos) const {
    return s.frames[pos / block_size] * block_size + pos % block_size;
  }

  int32_t take_frame() {
    int32_t f = free_list.pop_front();
    refs[f] = 1;
    return f;
  }

  void drop_ref(int32_t f) {
    if (refs[f] <= 0) return;  // already free: releasing again does nothing
    if (--refs[f] == 0) free_list.push_back(f);
  }

  // One append; on success fills *slot and the copy pair and records an undo entry.
  int append_one(int64_t id, int32_t* slot, int32_t* src, int32_t* dst, std::vector<Undo>* log) {
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
      u.taken = take_frame();
      s.frames.push_back(u.taken);
    } else {
      const int32_t tail = s.frames.back();
      if (refs[tail] > 1) {  // shared tail: move this writer onto a private copy
        if (free_list.size() == 0) return PA_ERR_OUT_OF_BLOCKS;
        u.kind = Undo::kCopyOnWrite;
        u.taken = take_frame();
        u.shared = tail;
        drop_ref(tail);
        s.frames.back() = u.taken;
        *src = tail;
        *dst = u.taken;
      }
    }
    s.len = t + 1;
    *slot = slot_of(s, t);
    if (log) log->push_back(u);
    return PA_OK;
  }

  void undo(const Undo& u) {
    Seq& s = seqs[u.seq];
    s.len -= 1;
    switch (u.kind) {
      case Undo::kInPlace:
        break;
      case Undo::kNewFrame:
        s.frames.pop_back();
        refs[u.taken] = 0;
        free_list.push_front(u.taken);
        break;
      case Undo::kCopyOnWrite:
        s.frames.back() = u.shared;
        refs[u.shared] += 1;
        refs[u.taken] = 0;
        free_list.push_front(u.taken);
        break;
    }
  }
};

extern "C" {

int pa_bm_create(int32_t num_blocks, int32_t block_size, const int32_t* free_order, pa_bm** bm_out) {
  if (!bm_out || num_blocks <= 0 || block_size <= 0) return PA_ERR_INVALID;
  if (static_cast<int64_t>(num_blocks) * block_size > INT32_MAX) return PA_ERR_INVALID;
  pa_bm* bm = new (std::nothrow) pa_bm();
  if (!bm) return PA_ERR_INVALID;
  bm->num_blocks = num_blocks;
  bm->block_size = block_size;
  bm->refs.assign(num_blocks, 0);
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
}

void pa_bm_destroy(pa_bm* bm) { delete bm; }

int pa_bm_add_seq(pa_bm* bm, int64_t seq_id, int32_t num_tokens, int32_t* slots_out) {
  if (!bm || num_tokens < 0) return PA_ERR_INVALID;
  if (bm->seqs.count(seq_id)) return PA_ERR_SEQ_EXISTS;
  const int32_t need = num_tokens / bm->block_size + (num_tokens % bm->block_size != 0);
  if (need > bm->free_list.size()) return PA_ERR_OUT_OF_BLOCKS;
  Seq s;
  s.frames.reserve(need + 1);
  for (int32_t j = 0; j < need; ++j) s.frames.push_back(bm->take_frame());
  s.len = num_tokens;
  if (slots_out)
    for (int32_t i = 0; i < num_tokens; ++i) slots_out[i] = bm->slot_of(s, i);
  bm->seqs.emplace(seq_id, std::move(s));
  return PA_OK;
}

int pa_bm_append(pa_bm* bm, int64_t seq_id, int32_t* slot_out, int32_t* cow_src, int32_t* cow_dst) {
  if (!bm || !slot_out) return PA_ERR_INVALID;
  int32_t src, dst;
  int rc = bm->append_one(seq_id, slot_out, &src, &dst, nullptr);
  if (rc != PA_OK) return rc;
  if (cow_src) *cow_src = src;
  if (cow_dst) *cow_dst = dst;
  return PA_OK;
}

int pa_bm_step(pa_bm* bm, const int64_t* seq_ids, int32_t n, int32_t* slots_out,
               int32_t* copies_out, int32_t* n_copies_out) {
  if (!bm || n < 0 || (n > 0 && (!seq_ids || !slots_out))) return PA_ERR_INVALID;
  std::vector<Undo> log;
  log.reserve(n);
  int32_t n_copies = 0;
  for (int32_t i = 0; i < n; ++i) {
    int32_t src, dst;
    int rc = bm->append_one(seq_ids[i], &slots_out[i], &src, &dst, &log);
    if (rc != PA_OK) {
      for (auto u = log.rbegin(); u != log.rend(); ++u) bm->undo(*u);
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

int pa_bm_extend(pa_bm* bm, int64_t seq_id, int32_t num_tokens, int32_t* slots_out, int32_t* copies_out,
                 int32_t* n_copies_out) {
  if (!bm || num_tokens < 0 || (num_tokens > 0 && !slots_out)) return PA_ERR_INVALID;
  if (!bm->seqs.count(seq_id)) return PA_ERR_UNKNOWN_SEQ;
  std::vector<Undo> log;
  log.reserve(num_tokens);
  int32_t n_copies = 0;
  for (int32_t i = 0; i < num_tokens; ++i) {
    int32_t src, dst;
    int rc = bm->append_one(seq_id, &slots_out[i], &src, &dst, &log);
    if (rc != PA_OK) {
      for (auto u = log.rbegin(); u != log.rend(); ++u) bm->undo(*u);
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

int pa_bm_fork(pa_bm* bm, int64_t parent_id, int64_t child_id) {
  if (!bm) return PA_ERR_INVALID;
  auto p = bm->seqs.find(parent_id);
  if (p == bm->seqs.end()) return PA_ERR_UNKNOWN_SEQ;
  if (bm->seqs.count(child_id)) return PA_ERR_SEQ_EXISTS;
  Seq child = p->second;  // copy of the table and the length
  for (int32_t f : child.frames) bm->refs[f] += 1;
  bm->seqs.emplace(child_id, std::move(child));
  return PA_OK;
}

int pa_bm_free(pa_bm* bm, int64_t seq_id) {
  if (!bm) return PA_ERR_INVALID;
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return PA_WARN_DOUBLE_FREE;
  for (int32_t f : it->second.frames) bm->drop_ref(f);
  bm->seqs.erase(it);
  return PA_OK;
}

int pa_bm_block_tables(const pa_bm* bm, const int64_t* seq_ids, int32_t n, int32_t max_blocks,
                       int32_t* tables_out, int32_t* lens_out) {
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
}

int pa_bm_seq_info(const pa_bm* bm, int64_t seq_id, int32_t* len_out, int32_t* n_blocks_out) {
  if (!bm) return PA_ERR_INVALID;
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return PA_ERR_UNKNOWN_SEQ;
  if (len_out) *len_out = it->second.len;
  if (n_blocks_out) *n_blocks_out = static_cast<int32_t>(it->second.frames.size());
  return PA_OK;
}

int pa_bm_table(const pa_bm* bm, int64_t seq_id, int32_t* out, int32_t cap, int32_t* n_out) {
  if (!bm || cap < 0 || (cap > 0 && !out)) return PA_ERR_INVALID;
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return PA_ERR_UNKNOWN_SEQ;
  const auto& fr = it->second.frames;
  if (n_out) *n_out = static_cast<int32_t>(fr.size());
  if (static_cast<int32_t>(fr.size()) > cap) return PA_ERR_CAPACITY;
  if (!fr.empty()) std::memcpy(out, fr.data(), sizeof(int32_t) * fr.size());
  return PA_OK;
}

int pa_bm_slot(const pa_bm* bm, int64_t seq_id, int32_t pos, int32_t* slot_out) {
  if (!bm || !slot_out) return PA_ERR_INVALID;
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return PA_ERR_UNKNOWN_SEQ;
  if (pos < 0 || pos >= it->second.len) return PA_ERR_INVALID;
  *slot_out = bm->slot_of(it->second, pos);
  return PA_OK;
}

int pa_bm_num_free(const pa_bm* bm, int32_t* n_out) {
  if (!bm || !n_out) return PA_ERR_INVALID;
  *n_out = bm->free_list.size();
  return PA_OK;
}

int pa_bm_free_list(const pa_bm* bm, int32_t* out, int32_t cap, int32_t* n_out) {
  if (!bm || cap < 0 || (cap > 0 && !out)) return PA_ERR_INVALID;
  const int32_t n = bm->free_list.size();
  if (n_out) *n_out = n;
  if (n > cap) return PA_ERR_CAPACITY;
  for (int32_t i = 0; i < n; ++i) out[i] = bm->free_list.at(i);
  return PA_OK;
}

int pa_bm_ref_counts(const pa_bm* bm, int32_t* out, int32_t cap) {
  if (!bm || !out) return PA_ERR_INVALID;
  if (cap < bm->num_blocks) return PA_ERR_CAPACITY;
  std::memcpy(out, bm->refs.data(), sizeof(int32_t) * bm->num_blocks);
  return PA_OK;
}

int pa_bm_num_seqs(const pa_bm* bm, int32_t* n_out) {
  if (!bm || !n_out) return PA_ERR_INVALID;
  *n_out = static_cast<int32_t>(bm->seqs.size());
  return PA_OK;
}

}  // extern "C"
