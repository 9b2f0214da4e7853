// Host-side block manager for the paged KV cache (C ABI in include/pkv.h).
//
// First page, section 4.2 ("paged KV cache and tiered CPU offload"): a block
// manager hands out fixed-size blocks on demand, allocate(seq, num_tokens)
// taking ceil(num_tokens / block_size) blocks from a free list, and a tiered
// manager keeps a sequence's most recent `gpu_window` blocks in the GPU pool
// while older blocks move to a pinned-CPU pool, coming back by DMA when
// needed.  Third page, "continuous batching": between two kernel launches the
// runtime updates this metadata for every sequence that joins, grows or
// leaves.  Shared prefixes (first page, section 1: exact-prefix reuse) are
// blocks referenced by several sequences; a sequence that writes into a
// shared block first gets its own copy (copy-on-write).
//
// The manager only does bookkeeping; the data moves with pkv_copy_blocks.
#include <cstdint>
#include <mutex>
#include <unordered_map>
#include <vector>

#include "pkv.h"

struct pkv_block_manager {
  int32_t block_size = 0;
  std::vector<int32_t> gpu_free, cpu_free;  // stacks of free block ids
  std::vector<int32_t> gpu_ref, cpu_ref;    // reference counts
  struct Seq {
    int32_t num_tokens = 0;
    std::vector<int32_t> blocks;   // logical block j -> id in its pool
    std::vector<uint8_t> on_cpu;   // 1 if block j lives in the CPU pool
  };
  std::unordered_map<int64_t, Seq> seqs;
  std::mutex mu;
};

namespace {

int32_t pop(std::vector<int32_t>& free_list, std::vector<int32_t>& ref) {
  const int32_t id = free_list.back();
  free_list.pop_back();
  ref[id] = 1;
  return id;
}

void release(std::vector<int32_t>& free_list, std::vector<int32_t>& ref, int32_t id) {
  if (--ref[id] == 0) free_list.push_back(id);
}

int32_t blocks_for(int64_t tokens, int32_t bs) {
  return static_cast<int32_t>((tokens + bs - 1) / bs);
}

}  // namespace

extern "C" pkv_block_manager* pkv_bm_create(int32_t num_gpu_blocks, int32_t num_cpu_blocks,
                                            int32_t block_size) {
  if (num_gpu_blocks < 0 || num_cpu_blocks < 0 || block_size < 1) return nullptr;
  auto* m = new pkv_block_manager;
  m->block_size = block_size;
  m->gpu_ref.assign(num_gpu_blocks, 0);
  m->cpu_ref.assign(num_cpu_blocks, 0);
  // Free lists are stacks: lowest ids come out first, later the most
  // recently freed block is reused first.
  for (int32_t i = num_gpu_blocks - 1; i >= 0; --i) m->gpu_free.push_back(i);
  for (int32_t i = num_cpu_blocks - 1; i >= 0; --i) m->cpu_free.push_back(i);
  return m;
}

extern "C" void pkv_bm_destroy(pkv_block_manager* m) { delete m; }

extern "C" int pkv_bm_add_sequence(pkv_block_manager* m, int64_t seq_id, int32_t num_tokens) {
  if (!m) return PKV_ERR_NULL;
  if (num_tokens < 0) return PKV_ERR_INVALID;
  std::lock_guard<std::mutex> lock(m->mu);
  if (m->seqs.count(seq_id)) return PKV_ERR_INVALID;
  const int32_t need = blocks_for(num_tokens, m->block_size);
  if (static_cast<size_t>(need) > m->gpu_free.size()) return PKV_ERR_NO_BLOCKS;
  pkv_block_manager::Seq s;
  s.num_tokens = num_tokens;
  for (int32_t j = 0; j < need; ++j) {
    s.blocks.push_back(pop(m->gpu_free, m->gpu_ref));
    s.on_cpu.push_back(0);
  }
  m->seqs.emplace(seq_id, std::move(s));
  return PKV_OK;
}

extern "C" int pkv_bm_fork(pkv_block_manager* m, int64_t parent, int64_t child) {
  if (!m) return PKV_ERR_NULL;
  std::lock_guard<std::mutex> lock(m->mu);
  auto it = m->seqs.find(parent);
  if (it == m->seqs.end() || m->seqs.count(child)) return PKV_ERR_INVALID;
  const pkv_block_manager::Seq& p = it->second;
  for (uint8_t c : p.on_cpu)
    if (c) return PKV_ERR_INVALID;  // swap the parent in first
  for (int32_t id : p.blocks) ++m->gpu_ref[id];
  pkv_block_manager::Seq s = p;
  m->seqs.emplace(child, std::move(s));
  return PKV_OK;
}

extern "C" int pkv_bm_append_token(pkv_block_manager* m, int64_t seq_id, int32_t* slot,
                                   int32_t* copy_src, int32_t* copy_dst) {
  if (!m || !slot || !copy_src || !copy_dst) return PKV_ERR_NULL;
  std::lock_guard<std::mutex> lock(m->mu);
  auto it = m->seqs.find(seq_id);
  if (it == m->seqs.end()) return PKV_ERR_INVALID;
  pkv_block_manager::Seq& s = it->second;
  const int32_t bs = m->block_size;
  const int32_t pos = s.num_tokens;
  *copy_src = *copy_dst = -1;
  if (pos % bs == 0) {
    if (m->gpu_free.empty()) return PKV_ERR_NO_BLOCKS;
    s.blocks.push_back(pop(m->gpu_free, m->gpu_ref));
    s.on_cpu.push_back(0);
  } else {
    const size_t j = s.blocks.size() - 1;
    if (s.on_cpu[j]) return PKV_ERR_INVALID;  // swap in first
    const int32_t old = s.blocks[j];
    if (m->gpu_ref[old] > 1) {
      // the block is shared: this sequence gets its own copy before writing
      if (m->gpu_free.empty()) return PKV_ERR_NO_BLOCKS;
      const int32_t fresh = pop(m->gpu_free, m->gpu_ref);
      --m->gpu_ref[old];
      s.blocks[j] = fresh;
      *copy_src = old;
      *copy_dst = fresh;
    }
  }
  *slot = s.blocks.back() * bs + pos % bs;
  s.num_tokens = pos + 1;
  return PKV_OK;
}

extern "C" int pkv_bm_free_sequence(pkv_block_manager* m, int64_t seq_id) {
  if (!m) return PKV_ERR_NULL;
  std::lock_guard<std::mutex> lock(m->mu);
  auto it = m->seqs.find(seq_id);
  if (it == m->seqs.end()) return PKV_ERR_INVALID;
  const pkv_block_manager::Seq& s = it->second;
  for (size_t j = 0; j < s.blocks.size(); ++j) {
    if (s.on_cpu[j])
      release(m->cpu_free, m->cpu_ref, s.blocks[j]);
    else
      release(m->gpu_free, m->gpu_ref, s.blocks[j]);
  }
  m->seqs.erase(it);
  return PKV_OK;
}

extern "C" int pkv_bm_swap_out(pkv_block_manager* m, int64_t seq_id, int32_t gpu_window,
                               int32_t* pairs, int32_t max_pairs, int32_t* num_pairs) {
  if (!m || !num_pairs || (max_pairs > 0 && !pairs)) return PKV_ERR_NULL;
  if (gpu_window < 0 || max_pairs < 0) return PKV_ERR_INVALID;
  std::lock_guard<std::mutex> lock(m->mu);
  auto it = m->seqs.find(seq_id);
  if (it == m->seqs.end()) return PKV_ERR_INVALID;
  pkv_block_manager::Seq& s = it->second;
  const int32_t nb = static_cast<int32_t>(s.blocks.size());
  // Cold blocks: everything before the last gpu_window blocks that is still
  // on the GPU and not shared with another sequence.
  std::vector<int32_t> cold;
  for (int32_t j = 0; j < nb - gpu_window; ++j)
    if (!s.on_cpu[j] && m->gpu_ref[s.blocks[j]] == 1) cold.push_back(j);
  if (static_cast<int32_t>(cold.size()) > max_pairs) return PKV_ERR_INVALID;
  if (cold.size() > m->cpu_free.size()) return PKV_ERR_NO_BLOCKS;
  for (size_t k = 0; k < cold.size(); ++k) {
    const int32_t j = cold[k];
    const int32_t g = s.blocks[j];
    const int32_t c = pop(m->cpu_free, m->cpu_ref);
    release(m->gpu_free, m->gpu_ref, g);
    s.blocks[j] = c;
    s.on_cpu[j] = 1;
    pairs[2 * k] = g;
    pairs[2 * k + 1] = c;
  }
  *num_pairs = static_cast<int32_t>(cold.size());
  return PKV_OK;
}

extern "C" int pkv_bm_swap_in(pkv_block_manager* m, int64_t seq_id, int32_t* pairs,
                              int32_t max_pairs, int32_t* num_pairs) {
  if (!m || !num_pairs || (max_pairs > 0 && !pairs)) return PKV_ERR_NULL;
  if (max_pairs < 0) return PKV_ERR_INVALID;
  std::lock_guard<std::mutex> lock(m->mu);
  auto it = m->seqs.find(seq_id);
  if (it == m->seqs.end()) return PKV_ERR_INVALID;
  pkv_block_manager::Seq& s = it->second;
  std::vector<int32_t> warm;
  for (size_t j = 0; j < s.blocks.size(); ++j)
    if (s.on_cpu[j]) warm.push_back(static_cast<int32_t>(j));
  if (static_cast<int32_t>(warm.size()) > max_pairs) return PKV_ERR_INVALID;
  if (warm.size() > m->gpu_free.size()) return PKV_ERR_NO_BLOCKS;
  for (size_t k = 0; k < warm.size(); ++k) {
    const int32_t j = warm[k];
    const int32_t c = s.blocks[j];
    const int32_t g = pop(m->gpu_free, m->gpu_ref);
    release(m->cpu_free, m->cpu_ref, c);
    s.blocks[j] = g;
    s.on_cpu[j] = 0;
    pairs[2 * k] = c;
    pairs[2 * k + 1] = g;
  }
  *num_pairs = static_cast<int32_t>(warm.size());
  return PKV_OK;
}

extern "C" int pkv_bm_num_free(pkv_block_manager* m, int32_t* gpu, int32_t* cpu) {
  if (!m || !gpu || !cpu) return PKV_ERR_NULL;
  std::lock_guard<std::mutex> lock(m->mu);
  *gpu = static_cast<int32_t>(m->gpu_free.size());
  *cpu = static_cast<int32_t>(m->cpu_free.size());
  return PKV_OK;
}

extern "C" int pkv_bm_seq_info(pkv_block_manager* m, int64_t seq_id, int32_t* num_tokens,
                               int32_t* num_blocks, int32_t* num_cpu_blocks) {
  if (!m || !num_tokens || !num_blocks || !num_cpu_blocks) return PKV_ERR_NULL;
  std::lock_guard<std::mutex> lock(m->mu);
  auto it = m->seqs.find(seq_id);
  if (it == m->seqs.end()) return PKV_ERR_INVALID;
  const pkv_block_manager::Seq& s = it->second;
  *num_tokens = s.num_tokens;
  *num_blocks = static_cast<int32_t>(s.blocks.size());
  int32_t c = 0;
  for (uint8_t x : s.on_cpu) c += x;
  *num_cpu_blocks = c;
  return PKV_OK;
}

extern "C" int pkv_bm_block_tables(pkv_block_manager* m, const int64_t* seq_ids, int32_t n,
                                   int32_t max_blocks_per_seq, int32_t* block_tables,
                                   int32_t* context_lens) {
  if (!m || (n > 0 && (!seq_ids || !block_tables || !context_lens))) return PKV_ERR_NULL;
  if (n < 0 || max_blocks_per_seq < 1) return PKV_ERR_INVALID;
  std::lock_guard<std::mutex> lock(m->mu);
  for (int32_t i = 0; i < n; ++i) {
    auto it = m->seqs.find(seq_ids[i]);
    if (it == m->seqs.end()) return PKV_ERR_INVALID;
    const pkv_block_manager::Seq& s = it->second;
    if (static_cast<int32_t>(s.blocks.size()) > max_blocks_per_seq) return PKV_ERR_INVALID;
    for (uint8_t c : s.on_cpu)
      if (c) return PKV_ERR_INVALID;  // a decode reads the GPU pool only
  }
  for (int32_t i = 0; i < n; ++i) {
    const pkv_block_manager::Seq& s = m->seqs.find(seq_ids[i])->second;
    int32_t* row = block_tables + static_cast<size_t>(i) * max_blocks_per_seq;
    for (int32_t j = 0; j < max_blocks_per_seq; ++j)
      row[j] = j < static_cast<int32_t>(s.blocks.size()) ? s.blocks[j] : -1;
    context_lens[i] = s.num_tokens;
  }
  return PKV_OK;
}
