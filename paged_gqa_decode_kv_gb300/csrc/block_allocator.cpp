// block_allocator.cpp -- host-side pool of physical KV blocks with reference
// counts, on-demand growth, prefix sharing and copy-on-write, plus a host
// check of block tables.
//
// Semantics ("Module 10: inference and serving", sections "Mapping logical
// positions to physical blocks" and "Share only identical state"; "Ch. 6
// Inference efficiency and serving", 6.4; "The math of Transformer
// inference", section 9, PagedAttention):
//   - a sequence takes one more block when it grows past a block boundary, so
//     at most bs - 1 of its slots are unused;
//   - forks reference the same prefix blocks; a count per block records how
//     many sequences use it; a block returns to the pool when its count drops
//     to zero;
//   - a write into a shared block first gets a private copy (copy-on-write);
//     the device copy itself is pgd_copy_blocks.
// Every operation is O(1) per block id (free ids live on a stack) and either
// succeeds completely or changes nothing.
#include <stdarg.h>
#include <stdio.h>

#include <new>
#include <string>
#include <unordered_map>
#include <vector>

#include "../../include/pgd.h"

struct pgd_alloc {
  std::vector<int32_t> ref;         // reference count per id
  std::vector<int32_t> free_stack;  // ids with ref == 0
};

namespace pgd {
// The per-thread detail string behind pgd_last_error_detail, shared by every
// entry point of the library.
static thread_local std::string t_detail;
void set_error_detail(const char *msg) { t_detail = msg; }
void clear_error_detail() { t_detail.clear(); }
const char *error_detail() { return t_detail.c_str(); }
}  // namespace pgd

namespace {
pgd_status afail(pgd_status s, const char *fmt, ...) {
  char buf[256];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  pgd::set_error_detail(buf);
  return s;
}

bool held(const pgd_alloc *a, int32_t id) {
  return id >= 0 && id < (int32_t)a->ref.size() && a->ref[id] > 0;
}

int32_t take_one(pgd_alloc *a) {
  const int32_t id = a->free_stack.back();
  a->free_stack.pop_back();
  a->ref[id] = 1;
  return id;
}

void drop_one(pgd_alloc *a, int32_t id) {
  if (--a->ref[id] == 0) a->free_stack.push_back(id);
}
}  // namespace

extern "C" {

pgd_status pgd_alloc_create(int32_t num_blocks, pgd_alloc **out) {
  if (!out) return afail(PGD_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (num_blocks <= 0) return afail(PGD_ERR_INVALID_ARG, "num_blocks = %d", num_blocks);
  pgd_alloc *a = new (std::nothrow) pgd_alloc;
  if (!a) return afail(PGD_ERR_INVALID_ARG, "out of host memory");
  a->ref.assign((size_t)num_blocks, 0);
  a->free_stack.resize((size_t)num_blocks);
  // Lowest ids on top, so a fresh pool hands out 0, 1, 2, ...
  for (int32_t i = 0; i < num_blocks; ++i) a->free_stack[(size_t)i] = num_blocks - 1 - i;
  *out = a;
  return PGD_OK;
}

void pgd_alloc_destroy(pgd_alloc *a) { delete a; }

pgd_status pgd_alloc_allocate(pgd_alloc *a, int32_t n, int32_t *ids_out) {
  if (!a || n < 0 || (n > 0 && !ids_out)) return afail(PGD_ERR_INVALID_ARG, "bad arguments");
  if ((size_t)n > a->free_stack.size())
    return afail(PGD_ERR_OUT_OF_BLOCKS, "%d blocks asked, %zu free", n, a->free_stack.size());
  for (int32_t i = 0; i < n; ++i) ids_out[i] = take_one(a);
  return PGD_OK;
}

pgd_status pgd_alloc_share(pgd_alloc *a, const int32_t *ids, int32_t n) {
  if (!a || n < 0 || (n > 0 && !ids)) return afail(PGD_ERR_INVALID_ARG, "bad arguments");
  for (int32_t i = 0; i < n; ++i)
    if (!held(a, ids[i])) return afail(PGD_ERR_BLOCK_STATE, "share of unheld block %d", ids[i]);
  for (int32_t i = 0; i < n; ++i) ++a->ref[ids[i]];
  return PGD_OK;
}

pgd_status pgd_alloc_release(pgd_alloc *a, const int32_t *ids, int32_t n) {
  if (!a || n < 0 || (n > 0 && !ids)) return afail(PGD_ERR_INVALID_ARG, "bad arguments");
  std::unordered_map<int32_t, int32_t> need;
  for (int32_t i = 0; i < n; ++i) {
    if (!held(a, ids[i])) return afail(PGD_ERR_BLOCK_STATE, "release of unheld block %d", ids[i]);
    if (++need[ids[i]] > a->ref[ids[i]])
      return afail(PGD_ERR_BLOCK_STATE, "block %d released more often than held", ids[i]);
  }
  for (int32_t i = 0; i < n; ++i) drop_one(a, ids[i]);
  return PGD_OK;
}

int32_t pgd_alloc_refcount(const pgd_alloc *a, int32_t id) {
  if (!a || id < 0 || id >= (int32_t)a->ref.size()) return -1;
  return a->ref[id];
}

int32_t pgd_alloc_num_free(const pgd_alloc *a) { return a ? (int32_t)a->free_stack.size() : 0; }

int32_t pgd_alloc_num_blocks(const pgd_alloc *a) { return a ? (int32_t)a->ref.size() : 0; }

pgd_status pgd_alloc_append_slot(pgd_alloc *a, int32_t *row, int32_t MB, int32_t bs,
                                 int32_t pos, int32_t *cow_src, int32_t *cow_dst) {
  if (!a || !row || !cow_src || !cow_dst || MB <= 0 || bs <= 0)
    return afail(PGD_ERR_INVALID_ARG, "bad arguments");
  *cow_src = *cow_dst = -1;
  if (pos < 0 || pos / bs >= MB) return afail(PGD_ERR_INVALID_ARG, "position %d outside row", pos);
  const int32_t j = pos / bs;
  if (row[j] < 0) {
    // A block is opened only at its first slot, right after the previous one.
    if (pos % bs != 0 || (j > 0 && row[j - 1] < 0))
      return afail(PGD_ERR_BLOCK_STATE, "gap in the table row before position %d", pos);
    if (a->free_stack.empty()) return afail(PGD_ERR_OUT_OF_BLOCKS, "no free block");
    row[j] = take_one(a);
    return PGD_OK;
  }
  const int32_t old = row[j];
  if (!held(a, old)) return afail(PGD_ERR_BLOCK_STATE, "row points at unheld block %d", old);
  if (a->ref[old] > 1) {
    if (a->free_stack.empty()) return afail(PGD_ERR_OUT_OF_BLOCKS, "no free block for copy");
    const int32_t fresh = take_one(a);
    row[j] = fresh;
    drop_one(a, old);
    *cow_src = old;
    *cow_dst = fresh;
  }
  return PGD_OK;
}

pgd_status pgd_alloc_fork(pgd_alloc *a, const int32_t *src_row, int32_t n_tokens, int32_t bs,
                          int32_t *dst_row, int32_t MB) {
  if (!a || !src_row || !dst_row || bs <= 0 || MB <= 0 || n_tokens < 0)
    return afail(PGD_ERR_INVALID_ARG, "bad arguments");
  const int32_t nblk = (int32_t)(((long long)n_tokens + bs - 1) / bs);
  if (nblk > MB) return afail(PGD_ERR_INVALID_ARG, "fork of %d tokens exceeds the row", n_tokens);
  for (int32_t j = 0; j < nblk; ++j)
    if (!held(a, src_row[j]))
      return afail(PGD_ERR_BLOCK_STATE, "fork source block %d is not held", src_row[j]);
  for (int32_t j = 0; j < nblk; ++j) {
    ++a->ref[src_row[j]];
    dst_row[j] = src_row[j];
  }
  return PGD_OK;
}

pgd_status pgd_validate_tables(const int32_t *tables, const int32_t *lens, int32_t B, int32_t MB,
                               int32_t NB, int32_t bs) {
  if (B < 0 || MB <= 0 || NB <= 0 || bs <= 0 || (B > 0 && (!tables || !lens)))
    return afail(PGD_ERR_INVALID_ARG, "bad arguments");
  for (int32_t b = 0; b < B; ++b) {
    const long long c = lens[b];
    if (c < 1 || c > (long long)MB * bs)
      return afail(PGD_ERR_INVALID_ARG, "context_lens[%d] = %lld outside [1, %lld]", b, c,
                   (long long)MB * bs);
    const int32_t nblk = (int32_t)((c + bs - 1) / bs);
    for (int32_t j = 0; j < nblk; ++j) {
      const int32_t id = tables[(size_t)b * MB + j];
      if (id < 0 || id >= NB)
        return afail(PGD_ERR_INVALID_ARG, "block_tables[%d][%d] = %d outside [0, %d)", b, j, id,
                     NB);
    }
  }
  return PGD_OK;
}

}  // extern "C"
