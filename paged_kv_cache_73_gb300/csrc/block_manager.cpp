// Host block manager: block tables, FIFO free list, reference counts, copy-on-write.
//
// Rules from [note] "vLLM / PagedAttention -- 把 LLM 服务的瓶颈从显存碎片里救出来",
// sections 关键设计 2 (block table, on-demand allocation) and 关键设计 3 (sharing,
// reference counts, copy-on-write); [lecture] "vLLM", sections PagedAttention 原理
// (single-request walk-through) and Parallel Sampling 场景; [guide] "vLLM /
// PagedAttention (SOSP 2023)", sections 03 and 04 (shared prefix, step 4).
//
// Every mutating call checks everything it needs (ids, free-block count) before
// it changes anything, so a failing call leaves the state as it was.
#include <cstdint>
#include <cstring>
#include <deque>
#include <new>
#include <string>
#include <unordered_map>
#include <vector>

#include "pkv_internal.h"

namespace {

struct Logical {
  int32_t phys;
  int32_t filled;
};

struct Manager {
  int num_blocks = 0;
  int B = 0;
  std::deque<int32_t> free_list;
  std::vector<int32_t> ref;
  std::unordered_map<int64_t, std::vector<Logical>> seqs;
  std::unordered_map<int64_t, std::vector<Logical>> prefixes;
  int64_t cow_copies = 0;
  // event counters: sequences added on a registered prefix and the block references they took
  // from it; groups and blocks that left this manager (swapped away) or arrived (swapped in)
  int64_t prefix_seqs = 0, prefix_blocks = 0;
  int64_t groups_out = 0, blocks_out = 0, groups_in = 0, blocks_in = 0;

  int32_t take() {
    int32_t b = free_list.front();
    free_list.pop_front();
    ref[b] = 1;
    return b;
  }
  void release(int32_t b) {
    if (--ref[b] == 0) free_list.push_back(b);
  }
  // Blocks for `len` fresh tokens, filled left to right; caller checked the count.
  std::vector<Logical> fresh(int len) {
    int n = (len + B - 1) / B;
    std::vector<Logical> out;
    out.reserve(n);
    for (int j = 0; j < n; ++j) {
      int f = len - j * B < B ? len - j * B : B;
      out.push_back({take(), f});
    }
    return out;
  }
  void slots_of(const std::vector<Logical>& blocks, int64_t* out) const {
    int64_t k = 0;
    for (const Logical& lb : blocks)
      for (int r = 0; r < lb.filled; ++r) out[k++] = (int64_t)lb.phys * B + r;
  }
  // What one append to `blocks` will need, given `extra_dec` references already
  // given up on the last block by earlier appends in the same batch.
  bool needs_block(const std::vector<Logical>& blocks, int extra_dec) const {
    const Logical& last = blocks.back();
    if (last.filled == B) return true;
    return ref[last.phys] - extra_dec > 1;
  }
  // Free blocks that n >= 0 appends to `blocks` take: a copy of a shared partly filled last
  // block (the first append), then a new block each time the last one is full.
  int blocks_for_appends(const std::vector<Logical>& blocks, int n) const {
    if (n <= 0) return 0;
    const Logical& last = blocks.back();
    const int room = B - last.filled;                  // rows left in the last block
    const int copy = (room > 0 && ref[last.phys] > 1) ? 1 : 0;
    const int past = n - room;                         // tokens that spill into new blocks
    return copy + (past > 0 ? (past + B - 1) / B : 0);
  }
  // n appends in order (the caller checked the free blocks): slots to slots_out[0..n), the one
  // possible copy to cow_pair_out[0..2) with *num_cow = 0 or 1.
  void extend(std::vector<Logical>& blocks, int n, int64_t* slots_out, int64_t* cow_pair_out, int* num_cow) {
    int c = 0;
    for (int i = 0; i < n; ++i) {
      int32_t s, d;
      const int64_t slot = append(blocks, &s, &d);
      if (slots_out) slots_out[i] = slot;
      if (s >= 0) {
        if (cow_pair_out) {
          cow_pair_out[0] = s;
          cow_pair_out[1] = d;
        }
        ++c;
      }
    }
    if (num_cow) *num_cow = c;
  }
  // One append; the caller checked that a free block exists if one is needed.
  int64_t append(std::vector<Logical>& blocks, int32_t* src, int32_t* dst) {
    *src = -1;
    *dst = -1;
    Logical* last = &blocks.back();
    if (last->filled == B) {
      // the last block is full: the token opens a new logical block
      blocks.push_back({take(), 0});
      last = &blocks.back();
    } else if (ref[last->phys] > 1) {
      // shared and partly filled: move this sequence onto a copy
      int32_t nb = take();
      *src = last->phys;
      *dst = nb;
      ref[last->phys] -= 1;
      last->phys = nb;
      cow_copies += 1;
    }
    int64_t slot = (int64_t)last->phys * B + last->filled;
    last->filled += 1;
    return slot;
  }
};

constexpr int kBmCounters = 7;

Manager* M(pkv_bm* bm) { return reinterpret_cast<Manager*>(bm); }
const Manager* M(const pkv_bm* bm) { return reinterpret_cast<const Manager*>(bm); }

int oom(const Manager* m, int need) {
  return pkv::fail(PKV_ERR_OOM, "block manager: need %d free blocks, have %d", need,
                   (int)m->free_list.size());
}

}  // namespace

extern "C" {

pkv_bm* pkv_bm_create(int num_blocks, int block_size, const int32_t* free_order) {
  if (num_blocks <= 0 || block_size <= 0) {
    pkv::fail(PKV_ERR_INVALID_ARG, "pkv_bm_create: num_blocks=%d block_size=%d must be positive",
              num_blocks, block_size);
    return nullptr;
  }
  Manager* m = new (std::nothrow) Manager();
  if (!m) {
    pkv::fail(PKV_ERR_OOM, "pkv_bm_create: out of host memory");
    return nullptr;
  }
  m->num_blocks = num_blocks;
  m->B = block_size;
  m->ref.assign(num_blocks, 0);
  if (free_order) {
    std::vector<char> seen(num_blocks, 0);
    for (int i = 0; i < num_blocks; ++i) {
      int32_t b = free_order[i];
      if (b < 0 || b >= num_blocks || seen[b]) {
        delete m;
        pkv::fail(PKV_ERR_INVALID_ARG, "pkv_bm_create: free_order is not a permutation (entry %d = %d)", i, b);
        return nullptr;
      }
      seen[b] = 1;
      m->free_list.push_back(b);
    }
  } else {
    for (int i = 0; i < num_blocks; ++i) m->free_list.push_back(i);
  }
  return reinterpret_cast<pkv_bm*>(m);
}

void pkv_bm_destroy(pkv_bm* bm) { delete M(bm); }

int pkv_bm_add_seq(pkv_bm* bm, int64_t seq_id, int prompt_len, int64_t* slots_out) {
  if (!bm) return pkv::fail(PKV_ERR_INVALID_ARG, "pkv_bm_add_seq: null manager");
  Manager* m = M(bm);
  if (prompt_len <= 0) return pkv::fail(PKV_ERR_INVALID_ARG, "pkv_bm_add_seq: prompt_len=%d", prompt_len);
  if (m->seqs.count(seq_id)) return pkv::fail(PKV_ERR_INVALID_ARG, "pkv_bm_add_seq: sequence %lld exists", (long long)seq_id);
  int need = (prompt_len + m->B - 1) / m->B;
  if (need > (int)m->free_list.size()) return oom(m, need);
  auto& blocks = m->seqs[seq_id];
  blocks = m->fresh(prompt_len);
  if (slots_out) m->slots_of(blocks, slots_out);
  return PKV_OK;
}

int pkv_bm_fork(pkv_bm* bm, int64_t parent, int64_t child) {
  if (!bm) return pkv::fail(PKV_ERR_INVALID_ARG, "pkv_bm_fork: null manager");
  Manager* m = M(bm);
  auto it = m->seqs.find(parent);
  if (it == m->seqs.end()) return pkv::fail(PKV_ERR_NOT_FOUND, "pkv_bm_fork: no sequence %lld", (long long)parent);
  if (m->seqs.count(child)) return pkv::fail(PKV_ERR_INVALID_ARG, "pkv_bm_fork: sequence %lld exists", (long long)child);
  std::vector<Logical> copy = it->second;
  for (const Logical& lb : copy) m->ref[lb.phys] += 1;
  m->seqs.emplace(child, std::move(copy));
  return PKV_OK;
}

int pkv_bm_append_slot(pkv_bm* bm, int64_t seq_id, int64_t* slot, int32_t* cow_src, int32_t* cow_dst) {
  if (!bm || !slot || !cow_src || !cow_dst) return pkv::fail(PKV_ERR_INVALID_ARG, "pkv_bm_append_slot: null argument");
  Manager* m = M(bm);
  auto it = m->seqs.find(seq_id);
  if (it == m->seqs.end()) return pkv::fail(PKV_ERR_NOT_FOUND, "pkv_bm_append_slot: no sequence %lld", (long long)seq_id);
  if (m->needs_block(it->second, 0) && m->free_list.empty()) return oom(m, 1);
  *slot = m->append(it->second, cow_src, cow_dst);
  return PKV_OK;
}

int pkv_bm_append_slots(pkv_bm* bm, const int64_t* seq_ids, int n, int64_t* slots_out,
                        int64_t* cow_pairs_out, int* num_cow) {
  if (!bm || n < 0 || (n > 0 && (!seq_ids || !slots_out || !cow_pairs_out)) || !num_cow)
    return pkv::fail(PKV_ERR_INVALID_ARG, "pkv_bm_append_slots: bad argument");
  Manager* m = M(bm);
  std::vector<std::vector<Logical>*> lists(n);
  std::unordered_map<int64_t, int> seen;
  std::unordered_map<int32_t, int> dec;  // references given up on a block earlier in this batch
  int need = 0;
  for (int i = 0; i < n; ++i) {
    auto it = m->seqs.find(seq_ids[i]);
    if (it == m->seqs.end())
      return pkv::fail(PKV_ERR_NOT_FOUND, "pkv_bm_append_slots: no sequence %lld", (long long)seq_ids[i]);
    if (seen.count(seq_ids[i]))
      return pkv::fail(PKV_ERR_INVALID_ARG, "pkv_bm_append_slots: sequence %lld listed twice", (long long)seq_ids[i]);
    seen[seq_ids[i]] = 1;
    lists[i] = &it->second;
    const Logical& last = it->second.back();
    int d = dec.count(last.phys) ? dec[last.phys] : 0;
    if (m->needs_block(it->second, d)) {
      need += 1;
      if (last.filled != m->B) dec[last.phys] = d + 1;  // a copy gives up one reference
    }
  }
  if (need > (int)m->free_list.size()) return oom(m, need);
  int c = 0;
  for (int i = 0; i < n; ++i) {
    int32_t s, d;
    slots_out[i] = m->append(*lists[i], &s, &d);
    if (s >= 0) {
      cow_pairs_out[2 * c] = s;
      cow_pairs_out[2 * c + 1] = d;
      ++c;
    }
  }
  *num_cow = c;
  return PKV_OK;
}

int pkv_bm_free(pkv_bm* bm, int64_t seq_id) {
  if (!bm) return pkv::fail(PKV_ERR_INVALID_ARG, "pkv_bm_free: null manager");
  Manager* m = M(bm);
  auto it = m->seqs.find(seq_id);
  if (it == m->seqs.end()) return pkv::fail(PKV_ERR_NOT_FOUND, "pkv_bm_free: no sequence %lld", (long long)seq_id);
  for (const Logical& lb : it->second) m->release(lb.phys);
  m->seqs.erase(it);
  return PKV_OK;
}

int pkv_bm_register_prefix(pkv_bm* bm, int64_t prefix_id, int len, int64_t* slots_out) {
  if (!bm) return pkv::fail(PKV_ERR_INVALID_ARG, "pkv_bm_register_prefix: null manager");
  Manager* m = M(bm);
  if (len <= 0) return pkv::fail(PKV_ERR_INVALID_ARG, "pkv_bm_register_prefix: len=%d", len);
  if (m->prefixes.count(prefix_id))
    return pkv::fail(PKV_ERR_INVALID_ARG, "pkv_bm_register_prefix: prefix %lld exists", (long long)prefix_id);
  int need = (len + m->B - 1) / m->B;
  if (need > (int)m->free_list.size()) return oom(m, need);
  auto& blocks = m->prefixes[prefix_id];
  blocks = m->fresh(len);
  if (slots_out) m->slots_of(blocks, slots_out);
  return PKV_OK;
}

int pkv_bm_add_seq_with_prefix(pkv_bm* bm, int64_t seq_id, int64_t prefix_id, int suffix_len, int64_t* slots_out,
                               int64_t* cow_pair_out, int* num_cow) {
  if (!bm) return pkv::fail(PKV_ERR_INVALID_ARG, "pkv_bm_add_seq_with_prefix: null manager");
  if (suffix_len < 0 || (suffix_len > 0 && !slots_out))
    return pkv::fail(PKV_ERR_INVALID_ARG, "pkv_bm_add_seq_with_prefix: suffix_len=%d (slots_out %s)", suffix_len,
                     slots_out ? "given" : "null");
  Manager* m = M(bm);
  auto it = m->prefixes.find(prefix_id);
  if (it == m->prefixes.end())
    return pkv::fail(PKV_ERR_NOT_FOUND, "pkv_bm_add_seq_with_prefix: no prefix %lld", (long long)prefix_id);
  if (m->seqs.count(seq_id))
    return pkv::fail(PKV_ERR_INVALID_ARG, "pkv_bm_add_seq_with_prefix: sequence %lld exists", (long long)seq_id);
  // the suffix's blocks, counted as if the sequence already held its reference on every prefix
  // block: a partly filled last prefix block is then shared, so the first suffix token copies it
  std::vector<Logical> copy = it->second;
  int need = 0;
  if (suffix_len > 0) {
    const Logical& last = copy.back();
    const int room = m->B - last.filled;
    const int past = suffix_len - room;
    need = (room > 0 ? 1 : 0) + (past > 0 ? (past + m->B - 1) / m->B : 0);
  }
  if (need > (int)m->free_list.size()) return oom(m, need);
  for (const Logical& lb : copy) m->ref[lb.phys] += 1;
  m->prefix_seqs += 1;
  m->prefix_blocks += (int64_t)copy.size();
  auto& blocks = m->seqs.emplace(seq_id, std::move(copy)).first->second;
  m->extend(blocks, suffix_len, slots_out, cow_pair_out, num_cow);
  if (suffix_len == 0 && num_cow) *num_cow = 0;
  return PKV_OK;
}

int pkv_bm_extend(pkv_bm* bm, int64_t seq_id, int n, int64_t* slots_out, int64_t* cow_pair_out, int* num_cow) {
  if (!bm || n < 0 || (n > 0 && !slots_out))
    return pkv::fail(PKV_ERR_INVALID_ARG, "pkv_bm_extend: bad argument (n=%d)", n);
  Manager* m = M(bm);
  auto it = m->seqs.find(seq_id);
  if (it == m->seqs.end()) return pkv::fail(PKV_ERR_NOT_FOUND, "pkv_bm_extend: no sequence %lld", (long long)seq_id);
  const int need = m->blocks_for_appends(it->second, n);
  if (need > (int)m->free_list.size()) return oom(m, need);
  m->extend(it->second, n, slots_out, cow_pair_out, num_cow);
  if (n == 0 && num_cow) *num_cow = 0;
  return PKV_OK;
}

int pkv_bm_drop_prefix(pkv_bm* bm, int64_t prefix_id) {
  if (!bm) return pkv::fail(PKV_ERR_INVALID_ARG, "pkv_bm_drop_prefix: null manager");
  Manager* m = M(bm);
  auto it = m->prefixes.find(prefix_id);
  if (it == m->prefixes.end())
    return pkv::fail(PKV_ERR_NOT_FOUND, "pkv_bm_drop_prefix: no prefix %lld", (long long)prefix_id);
  for (const Logical& lb : it->second) m->release(lb.phys);
  m->prefixes.erase(it);
  return PKV_OK;
}

int pkv_bm_block_table(const pkv_bm* bm, int64_t seq_id, int32_t* out, int cap, int* n_blocks, int* ctx_len) {
  if (!bm || !n_blocks || !ctx_len || cap < 0 || (cap > 0 && !out))
    return pkv::fail(PKV_ERR_INVALID_ARG, "pkv_bm_block_table: bad argument");
  const Manager* m = M(bm);
  auto it = m->seqs.find(seq_id);
  if (it == m->seqs.end()) return pkv::fail(PKV_ERR_NOT_FOUND, "pkv_bm_block_table: no sequence %lld", (long long)seq_id);
  const auto& blocks = it->second;
  if ((int)blocks.size() > cap)
    return pkv::fail(PKV_ERR_INVALID_ARG, "pkv_bm_block_table: %d blocks exceed cap %d", (int)blocks.size(), cap);
  int ctx = 0;
  for (size_t j = 0; j < blocks.size(); ++j) {
    out[j] = blocks[j].phys;
    ctx += blocks[j].filled;
  }
  *n_blocks = (int)blocks.size();
  *ctx_len = ctx;
  return PKV_OK;
}

int pkv_bm_block_tables(const pkv_bm* bm, const int64_t* seq_ids, int n, int32_t* tables_out, int max_blocks,
                        int32_t* ctx_lens_out) {
  if (!bm || n < 0 || max_blocks <= 0 || (n > 0 && (!seq_ids || !tables_out || !ctx_lens_out)))
    return pkv::fail(PKV_ERR_INVALID_ARG, "pkv_bm_block_tables: bad argument");
  const Manager* m = M(bm);
  for (int i = 0; i < n; ++i) {
    auto it = m->seqs.find(seq_ids[i]);
    if (it == m->seqs.end())
      return pkv::fail(PKV_ERR_NOT_FOUND, "pkv_bm_block_tables: no sequence %lld", (long long)seq_ids[i]);
    if ((int)it->second.size() > max_blocks)
      return pkv::fail(PKV_ERR_INVALID_ARG, "pkv_bm_block_tables: sequence %lld has %d blocks > %d",
                       (long long)seq_ids[i], (int)it->second.size(), max_blocks);
  }
  for (int i = 0; i < n; ++i) {
    const auto& blocks = m->seqs.find(seq_ids[i])->second;
    int32_t* row = tables_out + (size_t)i * max_blocks;
    int ctx = 0;
    for (int j = 0; j < max_blocks; ++j) row[j] = j < (int)blocks.size() ? blocks[j].phys : -1;
    for (const Logical& lb : blocks) ctx += lb.filled;
    ctx_lens_out[i] = ctx;
  }
  return PKV_OK;
}

int pkv_bm_beam_step(pkv_bm* bm, const int64_t* parents, const int64_t* children, int k, const int64_t* retire,
                     int n_retire, int64_t* slots_out, int64_t* cow_pairs_out, int* num_cow) {
  if (!bm || k < 0 || n_retire < 0 || (k > 0 && (!parents || !children || !slots_out || !cow_pairs_out)) ||
      (n_retire > 0 && !retire) || !num_cow)
    return pkv::fail(PKV_ERR_INVALID_ARG, "pkv_bm_beam_step: bad argument");
  Manager* m = M(bm);
  std::unordered_map<int64_t, int> seen;
  for (int i = 0; i < k; ++i) {
    if (!m->seqs.count(parents[i]))
      return pkv::fail(PKV_ERR_NOT_FOUND, "pkv_bm_beam_step: no parent sequence %lld", (long long)parents[i]);
    if (m->seqs.count(children[i]) || seen.count(children[i]))
      return pkv::fail(PKV_ERR_INVALID_ARG, "pkv_bm_beam_step: child %lld exists or is listed twice",
                       (long long)children[i]);
    seen[children[i]] = 1;
  }
  std::unordered_map<int64_t, int> retired;
  for (int i = 0; i < n_retire; ++i) {
    if (!m->seqs.count(retire[i]))
      return pkv::fail(PKV_ERR_NOT_FOUND, "pkv_bm_beam_step: no retired sequence %lld", (long long)retire[i]);
    if (retired.count(retire[i]))
      return pkv::fail(PKV_ERR_INVALID_ARG, "pkv_bm_beam_step: sequence %lld retired twice", (long long)retire[i]);
    retired[retire[i]] = 1;
  }
  // Reference counts after the forks and frees, and the blocks those frees return.
  std::unordered_map<int32_t, int> delta;
  for (int i = 0; i < k; ++i)
    for (const Logical& lb : m->seqs[parents[i]]) delta[lb.phys] += 1;
  for (int i = 0; i < n_retire; ++i)
    for (const Logical& lb : m->seqs[retire[i]]) delta[lb.phys] -= 1;
  int returned = 0;
  for (const auto& kv : delta)
    if (m->ref[kv.first] > 0 && m->ref[kv.first] + kv.second == 0) ++returned;
  // Blocks the appends will take: one per child whose last block is full or still shared.
  std::unordered_map<int32_t, int> dec;
  int need = 0;
  for (int i = 0; i < k; ++i) {
    const Logical& last = m->seqs[parents[i]].back();
    if (last.filled == m->B) {
      ++need;
    } else {
      const int r = m->ref[last.phys] + delta[last.phys] - dec[last.phys];
      if (r > 1) {
        ++need;
        dec[last.phys] += 1;
      }
    }
  }
  if (need > (int)m->free_list.size() + returned) return oom(m, need - returned);
  for (int i = 0; i < k; ++i) {
    std::vector<Logical> copy = m->seqs[parents[i]];
    for (const Logical& lb : copy) m->ref[lb.phys] += 1;
    m->seqs.emplace(children[i], std::move(copy));
  }
  for (int i = 0; i < n_retire; ++i) {
    auto it = m->seqs.find(retire[i]);
    for (const Logical& lb : it->second) m->release(lb.phys);
    m->seqs.erase(it);
  }
  int c = 0;
  for (int i = 0; i < k; ++i) {
    int32_t src, dst;
    slots_out[i] = m->append(m->seqs[children[i]], &src, &dst);
    if (src >= 0) {
      cow_pairs_out[2 * c] = src;
      cow_pairs_out[2 * c + 1] = dst;
      ++c;
    }
  }
  *num_cow = c;
  return PKV_OK;
}

int pkv_bm_swap(pkv_bm* src_bm, pkv_bm* dst_bm, const int64_t* seq_ids, int n, int64_t* pairs_out, int cap_pairs,
                int* n_pairs) {
  // [lecture] 调度和抢占 (Swapping), [guide] 05: a preempted group leaves one pool whole and
  // comes back whole; every check comes before the first change.
  if (!src_bm || !dst_bm || src_bm == dst_bm)
    return pkv::fail(PKV_ERR_INVALID_ARG, "pkv_bm_swap: two distinct managers needed");
  Manager* src = M(src_bm);
  Manager* dst = M(dst_bm);
  if (src->B != dst->B)
    return pkv::fail(PKV_ERR_INVALID_ARG, "pkv_bm_swap: block sizes differ (%d, %d)", src->B, dst->B);
  if (n < 0 || (n > 0 && (!seq_ids || !n_pairs)) || cap_pairs < 0 || (cap_pairs > 0 && !pairs_out))
    return pkv::fail(PKV_ERR_INVALID_ARG, "pkv_bm_swap: bad arguments");
  std::unordered_map<int64_t, int> seen;
  for (int i = 0; i < n; ++i) {
    if (!seen.emplace(seq_ids[i], i).second)
      return pkv::fail(PKV_ERR_INVALID_ARG, "pkv_bm_swap: sequence %lld listed twice", (long long)seq_ids[i]);
    if (!src->seqs.count(seq_ids[i]))
      return pkv::fail(PKV_ERR_NOT_FOUND, "pkv_bm_swap: unknown sequence %lld", (long long)seq_ids[i]);
    if (dst->seqs.count(seq_ids[i]))
      return pkv::fail(PKV_ERR_INVALID_ARG, "pkv_bm_swap: sequence %lld exists on the destination",
                       (long long)seq_ids[i]);
  }
  // distinct blocks in order of first appearance, with the references the group holds
  std::unordered_map<int32_t, int> held;
  std::vector<int32_t> order;
  for (int i = 0; i < n; ++i) {
    for (const Logical& lb : src->seqs[seq_ids[i]]) {
      auto ins = held.emplace(lb.phys, 0);
      if (ins.second) order.push_back(lb.phys);
      ins.first->second += 1;
    }
  }
  for (int32_t b : order)
    if (held[b] != src->ref[b])
      return pkv::fail(PKV_ERR_INVALID_ARG, "pkv_bm_swap: block %d is also held outside the group", b);
  if ((int)order.size() > (int)dst->free_list.size()) return oom(dst, (int)order.size());
  if ((int)order.size() > cap_pairs)
    return pkv::fail(PKV_ERR_INVALID_ARG, "pkv_bm_swap: %d block moves, room for %d", (int)order.size(), cap_pairs);
  std::unordered_map<int32_t, int32_t> moved;
  for (size_t i = 0; i < order.size(); ++i) {
    const int32_t b = order[i];
    const int32_t nb = dst->take();
    dst->ref[nb] = src->ref[b];
    moved[b] = nb;
    pairs_out[2 * i] = b;
    pairs_out[2 * i + 1] = nb;
  }
  for (int i = 0; i < n; ++i) {
    auto it = src->seqs.find(seq_ids[i]);
    std::vector<Logical> blocks = std::move(it->second);
    src->seqs.erase(it);
    for (Logical& lb : blocks) lb.phys = moved[lb.phys];
    dst->seqs.emplace(seq_ids[i], std::move(blocks));
  }
  for (int32_t b : order) {
    src->ref[b] = 0;
    src->free_list.push_back(b);
  }
  if (n > 0) {
    src->groups_out += 1;
    dst->groups_in += 1;
  }
  src->blocks_out += (int64_t)order.size();
  dst->blocks_in += (int64_t)order.size();
  if (n_pairs) *n_pairs = (int)order.size();
  return PKV_OK;
}

int pkv_bm_ref_histogram(const pkv_bm* bm, int64_t* hist, int cap) {
  if (!bm || !hist || cap <= 0) return pkv::fail(PKV_ERR_INVALID_ARG, "pkv_bm_ref_histogram: bad arguments");
  const Manager* m = M(bm);
  for (int r = 0; r < cap; ++r) hist[r] = 0;
  for (int32_t c : m->ref) hist[c < cap - 1 ? c : cap - 1] += 1;
  return PKV_OK;
}

int pkv_bm_counters(const pkv_bm* bm, int64_t* out, int n) {
  if (!bm || !out || n < 0) return pkv::fail(PKV_ERR_INVALID_ARG, "pkv_bm_counters: bad arguments");
  const Manager* m = M(bm);
  const int64_t all[kBmCounters] = {m->cow_copies, m->prefix_seqs, m->prefix_blocks, m->groups_out,
                                    m->blocks_out, m->groups_in,   m->blocks_in};
  for (int i = 0; i < n && i < kBmCounters; ++i) out[i] = all[i];
  return n < kBmCounters ? n : kBmCounters;
}

int pkv_bm_ref_count(const pkv_bm* bm, int32_t block) {
  if (!bm) return pkv::fail(PKV_ERR_INVALID_ARG, "pkv_bm_ref_count: null manager");
  const Manager* m = M(bm);
  if (block < 0 || block >= m->num_blocks)
    return pkv::fail(PKV_ERR_INVALID_ARG, "pkv_bm_ref_count: block %d out of range", block);
  return m->ref[block];
}

int pkv_bm_stats(const pkv_bm* bm, int* free_blocks, int64_t* tail_waste_tokens, int64_t* cow_copies) {
  if (!bm) return pkv::fail(PKV_ERR_INVALID_ARG, "pkv_bm_stats: null manager");
  const Manager* m = M(bm);
  if (free_blocks) *free_blocks = (int)m->free_list.size();
  if (tail_waste_tokens) {
    int64_t w = 0;
    for (const auto& kv : m->seqs)
      for (const Logical& lb : kv.second) w += m->B - lb.filled;
    *tail_waste_tokens = w;
  }
  if (cow_copies) *cow_copies = m->cow_copies;
  return PKV_OK;
}

}  // extern "C"
