// pa_blocks.cu -- host-side block manager for the paged K/V pool, and the
// block-copy kernel its copy-on-write needs.
//
// The manager follows the block manager of the paged-attention-runtime design
// page: a free list of physical blocks, a reference count per block, and the
// list of blocks each sequence owns.  allocate / free_sequence /
// share_prefix / copy-on-write behave as that page describes: sharing a
// prefix raises the shared blocks' counts, writing into a shared block first
// moves the writer onto a fresh private block, and a block returns to the
// free list when its count reaches zero.  The tables it exports are the
// [B, max_blocks_per_seq] int32 block tables (-1 = unallocated) of the
// Hugging Face decoding path.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <new>
#include <vector>

#include "pagedgqa.h"

struct pa_block_manager {
  int32_t num_blocks;
  int32_t block_size;
  int32_t max_seqs;
  int32_t max_blocks_per_seq;
  std::vector<int32_t> free_list;  // stack: ids 0,1,2,... first, then the last freed
  std::vector<int32_t> refs;       // per physical block
  std::vector<std::vector<int32_t>> seqs;
  std::mutex mu;
};

namespace {

bool seq_ok(const pa_block_manager* m, int32_t s) { return m && s >= 0 && s < m->max_seqs; }

void release(pa_block_manager* m, int32_t blk) {
  if (--m->refs[blk] == 0) m->free_list.push_back(blk);
}

int32_t take(pa_block_manager* m) {
  const int32_t b = m->free_list.back();
  m->free_list.pop_back();
  m->refs[b] = 1;
  return b;
}

// cow_block with the manager's lock held.
int cow_locked(pa_block_manager* m, int32_t seq, int32_t index, int32_t* old_block,
               int32_t* new_block) {
  std::vector<int32_t>& s = m->seqs[seq];
  if (index < 0 || index >= (int32_t)s.size()) return PA_ERR_STATE;
  const int32_t b = s[index];
  if (m->refs[b] > 1 && m->free_list.empty()) return PA_ERR_NO_BLOCKS;
  *old_block = b;
  if (m->refs[b] == 1) {
    *new_block = b;  // private already: nothing to copy
    return PA_OK;
  }
  const int32_t nb = take(m);
  --m->refs[b];
  s[index] = nb;
  *new_block = nb;
  return PA_OK;
}

}  // namespace

extern "C" {

pa_block_manager* pa_bm_create(int32_t num_blocks, int32_t block_size, int32_t max_seqs,
                               int32_t max_blocks_per_seq) {
  if (num_blocks < 1 || block_size < 1 || max_seqs < 1 || max_blocks_per_seq < 1) return nullptr;
  pa_block_manager* m = new (std::nothrow) pa_block_manager;
  if (!m) return nullptr;
  m->num_blocks = num_blocks;
  m->block_size = block_size;
  m->max_seqs = max_seqs;
  m->max_blocks_per_seq = max_blocks_per_seq;
  m->free_list.resize(num_blocks);
  for (int32_t i = 0; i < num_blocks; ++i) m->free_list[i] = num_blocks - 1 - i;
  m->refs.assign(num_blocks, 0);
  m->seqs.resize(max_seqs);
  return m;
}

void pa_bm_destroy(pa_block_manager* m) { delete m; }

int pa_bm_allocate(pa_block_manager* m, int32_t seq, int32_t n) {
  if (!seq_ok(m, seq) || n < 0) return PA_ERR_STATE;
  std::lock_guard<std::mutex> lk(m->mu);
  std::vector<int32_t>& s = m->seqs[seq];
  if ((int64_t)s.size() + n > m->max_blocks_per_seq) return PA_ERR_STATE;
  if ((int64_t)m->free_list.size() < n) return PA_ERR_NO_BLOCKS;
  for (int32_t i = 0; i < n; ++i) s.push_back(take(m));
  return PA_OK;
}

int pa_bm_free_sequence(pa_block_manager* m, int32_t seq) {
  if (!seq_ok(m, seq)) return PA_ERR_STATE;
  std::lock_guard<std::mutex> lk(m->mu);
  for (int32_t b : m->seqs[seq]) release(m, b);
  m->seqs[seq].clear();
  return PA_OK;
}

int pa_bm_share_prefix(pa_block_manager* m, int32_t src, int32_t dst, int32_t n) {
  if (!seq_ok(m, src) || !seq_ok(m, dst) || src == dst || n < 0) return PA_ERR_STATE;
  std::lock_guard<std::mutex> lk(m->mu);
  const std::vector<int32_t>& s = m->seqs[src];
  std::vector<int32_t>& d = m->seqs[dst];
  if (!d.empty() || n > (int32_t)s.size()) return PA_ERR_STATE;
  for (int32_t i = 0; i < n; ++i) {
    d.push_back(s[i]);
    ++m->refs[s[i]];
  }
  return PA_OK;
}

int pa_bm_copy_on_write(pa_block_manager* m, int32_t seq, int32_t index, int32_t* old_block,
                        int32_t* new_block) {
  if (!seq_ok(m, seq) || !old_block || !new_block) return PA_ERR_STATE;
  std::lock_guard<std::mutex> lk(m->mu);
  return cow_locked(m, seq, index, old_block, new_block);
}

int pa_bm_reserve_slot(pa_block_manager* m, int32_t seq, int32_t pos, int32_t* old_block,
                       int32_t* new_block) {
  if (!seq_ok(m, seq) || pos < 0 || !old_block || !new_block) return PA_ERR_STATE;
  const int32_t idx = pos / m->block_size;
  std::lock_guard<std::mutex> lk(m->mu);
  std::vector<int32_t>& s = m->seqs[seq];
  if (idx > (int32_t)s.size() || idx >= m->max_blocks_per_seq) return PA_ERR_STATE;
  if (idx < (int32_t)s.size()) return cow_locked(m, seq, idx, old_block, new_block);
  if (m->free_list.empty()) return PA_ERR_NO_BLOCKS;
  s.push_back(take(m));
  *old_block = *new_block = s.back();
  return PA_OK;
}

int pa_bm_block_table(pa_block_manager* m, const int32_t* seq_ids, int32_t rows, int32_t cols,
                      int32_t* table) {
  if (!m || rows < 0 || cols < 0 || (rows > 0 && (!seq_ids || !table))) return PA_ERR_STATE;
  std::lock_guard<std::mutex> lk(m->mu);
  for (int32_t r = 0; r < rows; ++r) {
    const int32_t sid = seq_ids[r];
    if (sid < 0 || sid >= m->max_seqs) return PA_ERR_STATE;
    const std::vector<int32_t>& s = m->seqs[sid];
    if ((int32_t)s.size() > cols) return PA_ERR_STATE;
    for (int32_t c = 0; c < cols; ++c) table[(int64_t)r * cols + c] = c < (int32_t)s.size() ? s[c] : -1;
  }
  return PA_OK;
}

int pa_bm_query(pa_block_manager* m, int32_t what, int32_t arg) {
  if (!m) return PA_ERR_STATE;
  std::lock_guard<std::mutex> lk(m->mu);
  switch (what) {
    case PA_BM_FREE_BLOCKS: return (int)m->free_list.size();
    case PA_BM_REF_COUNT:
      return (arg >= 0 && arg < m->num_blocks) ? m->refs[arg] : PA_ERR_STATE;
    case PA_BM_SEQ_BLOCKS:
      return (arg >= 0 && arg < m->max_seqs) ? (int)m->seqs[arg].size() : PA_ERR_STATE;
    default: return PA_ERR_STATE;
  }
}

}  // extern "C"

// ------------------------------------------------------------ block copy

namespace {

// Copy whole physical blocks (all rows, all kv heads, K and V):
// block (pair p, chunk c) moves 16-byte units c*blockDim + tid, ... of pair p.
__global__ void pa_copy_blocks_kernel(uint4* k, uint4* v, const int32_t* pairs, int32_t n,
                                      int64_t units, int32_t P, uint32_t* status) {
  const int32_t p = blockIdx.y;
  if (p >= n) return;
  const int32_t src = __ldg(pairs + 2 * p), dst = __ldg(pairs + 2 * p + 1);
  if (src < 0 || src >= P || dst < 0 || dst >= P) {
    if (status && blockIdx.x == 0 && threadIdx.x == 0) atomicOr(status, PA_STATUS_BAD_BLOCK);
    return;
  }
  if (src == dst) return;
  for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < units;
       u += (int64_t)gridDim.x * blockDim.x) {
    k[(int64_t)dst * units + u] = k[(int64_t)src * units + u];
    v[(int64_t)dst * units + u] = v[(int64_t)src * units + u];
  }
}

}  // namespace

extern "C" int pa_copy_blocks(const pa_shape* shape, void* k_cache, void* v_cache,
                              const int32_t* pairs, int32_t n_pairs, uint32_t* status,
                              pa_stream_t stream) {
  if (!shape || !k_cache || !v_cache || (n_pairs > 0 && !pairs)) return PA_ERR_NULL;
  if (n_pairs < 0 || n_pairs > 65535 || shape->num_blocks < 1 || shape->block_size < 1 ||
      shape->num_kv_heads < 1 || shape->head_dim < 8 || shape->head_dim % 8 != 0)
    return PA_ERR_SHAPE;
  if ((reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache)) & 15u)
    return PA_ERR_ALIGN;
  if (n_pairs == 0) return PA_OK;
  const int64_t units = (int64_t)shape->block_size * shape->num_kv_heads * shape->head_dim / 8;
  int gx = (int)((units + 255) / 256);
  if (gx > 64) gx = 64;
  pa_copy_blocks_kernel<<<dim3(gx, n_pairs), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), pairs, n_pairs, units,
      shape->num_blocks, status);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}
