// pkv_block_manager.cpp -- host-side KV block allocator: the part of the scheduler that
// produces the block tables and slot mappings the kernels consume.
//
// "mini-vLLM" LLM-Inference-Engine README (architecture diagram and milestone M4): a
// Block Manager allocates physical blocks out of a fixed pool and keeps a block table
// per sequence; under memory pressure the most recently admitted sequence is preempted
// (LIFO).  "vLLM-Style Llama Inference Engine", How it works: the scheduler allocates
// physical KV-cache blocks, and finished requests release their blocks.
//
// Design: a LIFO stack of free block ids (a block freed last is handed out first), a
// hash map from sequence id to {length, blocks}, and the admission order for LIFO
// preemption.  Appending a token to a sequence allocates a new block only when the
// sequence's last block is full.  All operations are O(blocks touched); one mutex makes
// the manager safe to share between threads.
#include <algorithm>
#include <cstdint>
#include <mutex>
#include <new>
#include <unordered_map>
#include <vector>

#include "pkv_internal.h"

struct pkv_block_manager {
  struct Seq {
    int64_t len = 0;
    std::vector<int32_t> blocks;
    uint64_t order = 0;  // admission stamp (larger = more recent)
  };
  int64_t num_blocks = 0;
  int32_t block_size = 0;
  std::vector<int32_t> free_stack;  // top = back()
  std::unordered_map<int64_t, Seq> seqs;
  uint64_t stamp = 0;
  std::mutex mu;

  // Blocks a sequence of `len` tokens occupies.
  int64_t blocks_for(int64_t len) const { return (len + block_size - 1) / block_size; }

  void release(Seq &s) {
    for (auto it = s.blocks.rbegin(); it != s.blocks.rend(); ++it) free_stack.push_back(*it);
    s.blocks.clear();
  }
};

using pkv::set_error;

PKV_API pkv_block_manager *pkv_bm_create(int64_t num_blocks, int32_t block_size) {
  if (num_blocks <= 0 || num_blocks > 0x7fffffffLL || block_size <= 0) {
    set_error(PKV_ERR_SHAPE, "pkv_bm_create: need 0 < num_blocks < 2^31 and block_size > 0");
    return nullptr;
  }
  pkv_block_manager *m = new (std::nothrow) pkv_block_manager();
  if (!m) {
    set_error(PKV_ERR_NOSPACE, "pkv_bm_create: out of host memory");
    return nullptr;
  }
  m->num_blocks = num_blocks;
  m->block_size = block_size;
  m->free_stack.reserve((size_t)num_blocks);
  for (int64_t b = num_blocks - 1; b >= 0; --b) m->free_stack.push_back((int32_t)b);  // 0 first
  pkv::clear_error();
  return m;
}

PKV_API void pkv_bm_destroy(pkv_block_manager *m) { delete m; }

PKV_API int64_t pkv_bm_num_free_blocks(pkv_block_manager *m) {
  if (!m) return set_error(PKV_ERR_NULL, "pkv_bm_num_free_blocks: NULL manager");
  std::lock_guard<std::mutex> lk(m->mu);
  return (int64_t)m->free_stack.size();
}

PKV_API int pkv_bm_add_sequence(pkv_block_manager *m, int64_t seq_id, int64_t num_tokens) {
  if (!m) return set_error(PKV_ERR_NULL, "pkv_bm_add_sequence: NULL manager");
  if (num_tokens < 0) return set_error(PKV_ERR_SHAPE, "pkv_bm_add_sequence: num_tokens < 0");
  std::lock_guard<std::mutex> lk(m->mu);
  if (m->seqs.count(seq_id))
    return set_error(PKV_ERR_SHAPE, "pkv_bm_add_sequence: sequence %lld already present",
                     (long long)seq_id);
  const int64_t need = m->blocks_for(num_tokens);
  if (need > (int64_t)m->free_stack.size())
    return set_error(PKV_ERR_NOSPACE, "pkv_bm_add_sequence: %lld blocks needed, %zu free",
                     (long long)need, m->free_stack.size());
  pkv_block_manager::Seq s;
  s.len = num_tokens;
  s.order = ++m->stamp;
  s.blocks.reserve((size_t)need);
  for (int64_t i = 0; i < need; ++i) {
    s.blocks.push_back(m->free_stack.back());
    m->free_stack.pop_back();
  }
  m->seqs.emplace(seq_id, std::move(s));
  pkv::clear_error();
  return PKV_OK;
}

PKV_API int pkv_bm_append_slots(pkv_block_manager *m, const int64_t *seq_ids, int32_t n,
                                int64_t *slot_mapping) {
  if (!m || (n > 0 && (!seq_ids || !slot_mapping)))
    return set_error(PKV_ERR_NULL, "pkv_bm_append_slots: NULL argument");
  if (n < 0) return set_error(PKV_ERR_SHAPE, "pkv_bm_append_slots: n < 0");
  std::lock_guard<std::mutex> lk(m->mu);
  // all-or-nothing: check every sequence and count the new blocks first
  int64_t new_blocks = 0;
  std::unordered_map<int64_t, int64_t> extra;  // appends per sequence in this call
  for (int32_t i = 0; i < n; ++i) {
    auto it = m->seqs.find(seq_ids[i]);
    if (it == m->seqs.end())
      return set_error(PKV_ERR_SHAPE, "pkv_bm_append_slots: unknown sequence %lld",
                       (long long)seq_ids[i]);
    const int64_t pos = it->second.len + extra[seq_ids[i]]++;
    if (pos % m->block_size == 0 && pos / m->block_size >= (int64_t)it->second.blocks.size())
      ++new_blocks;
  }
  if (new_blocks > (int64_t)m->free_stack.size())
    return set_error(PKV_ERR_NOSPACE, "pkv_bm_append_slots: %lld new blocks needed, %zu free",
                     (long long)new_blocks, m->free_stack.size());
  for (int32_t i = 0; i < n; ++i) {
    pkv_block_manager::Seq &s = m->seqs[seq_ids[i]];
    const int64_t pos = s.len++;
    const int64_t lb = pos / m->block_size;
    if (lb >= (int64_t)s.blocks.size()) {
      s.blocks.push_back(m->free_stack.back());
      m->free_stack.pop_back();
    }
    slot_mapping[i] = (int64_t)s.blocks[(size_t)lb] * m->block_size + pos % m->block_size;
  }
  pkv::clear_error();
  return PKV_OK;
}

PKV_API int pkv_bm_free_sequence(pkv_block_manager *m, int64_t seq_id) {
  if (!m) return set_error(PKV_ERR_NULL, "pkv_bm_free_sequence: NULL manager");
  std::lock_guard<std::mutex> lk(m->mu);
  auto it = m->seqs.find(seq_id);
  if (it == m->seqs.end())
    return set_error(PKV_ERR_SHAPE, "pkv_bm_free_sequence: unknown sequence %lld",
                     (long long)seq_id);
  m->release(it->second);
  m->seqs.erase(it);
  pkv::clear_error();
  return PKV_OK;
}

PKV_API int pkv_bm_preempt_lifo(pkv_block_manager *m, int64_t *seq_id) {
  if (!m || !seq_id) return set_error(PKV_ERR_NULL, "pkv_bm_preempt_lifo: NULL argument");
  std::lock_guard<std::mutex> lk(m->mu);
  if (m->seqs.empty()) return set_error(PKV_ERR_NOSPACE, "pkv_bm_preempt_lifo: no sequence to preempt");
  auto victim = m->seqs.begin();
  for (auto it = m->seqs.begin(); it != m->seqs.end(); ++it)
    if (it->second.order > victim->second.order) victim = it;
  *seq_id = victim->first;
  m->release(victim->second);
  m->seqs.erase(victim);
  pkv::clear_error();
  return PKV_OK;
}

PKV_API int pkv_bm_block_tables(pkv_block_manager *m, const int64_t *seq_ids, int32_t n,
                                int32_t max_blocks_per_seq, int32_t *block_tables,
                                int32_t *context_lens) {
  if (!m || (n > 0 && (!seq_ids || !block_tables || !context_lens)))
    return set_error(PKV_ERR_NULL, "pkv_bm_block_tables: NULL argument");
  if (n < 0 || max_blocks_per_seq <= 0)
    return set_error(PKV_ERR_SHAPE, "pkv_bm_block_tables: bad sizes");
  std::lock_guard<std::mutex> lk(m->mu);
  for (int32_t i = 0; i < n; ++i) {
    auto it = m->seqs.find(seq_ids[i]);
    if (it == m->seqs.end())
      return set_error(PKV_ERR_SHAPE, "pkv_bm_block_tables: unknown sequence %lld",
                       (long long)seq_ids[i]);
    const std::vector<int32_t> &blk = it->second.blocks;
    if ((int64_t)blk.size() > max_blocks_per_seq)
      return set_error(PKV_ERR_SHAPE, "pkv_bm_block_tables: sequence %lld has %zu blocks > %d",
                       (long long)seq_ids[i], blk.size(), max_blocks_per_seq);
    if (it->second.len > 0x7fffffffLL)
      return set_error(PKV_ERR_UNSUPPORTED, "pkv_bm_block_tables: length over 2^31-1");
    int32_t *row = block_tables + (int64_t)i * max_blocks_per_seq;
    std::copy(blk.begin(), blk.end(), row);
    std::fill(row + blk.size(), row + max_blocks_per_seq, -1);
    context_lens[i] = (int32_t)it->second.len;
  }
  pkv::clear_error();
  return PKV_OK;
}
