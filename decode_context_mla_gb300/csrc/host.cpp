// Host half of libdcpmla: the shared virtual allocator, the request -> token
// map, the host position map and status strings.
//
// SGLang "Decode Context Parallelism" docs, Architecture > Virtual KV layout:
// one allocator serves all c ranks of a DCP group.  It hands out virtual pages
// of P*c tokens; virtual page g is physical page g (P tokens) on every rank, so
// a rank's write of its own positions lands compacted in that page.
#include <algorithm>
#include <cstring>
#include <deque>
#include <new>
#include <vector>

#include "dcpmla.h"

struct dcpmla_alloc {
  int32_t c = 1;
  int32_t P = 1;
  int64_t num_pages = 0;
  std::deque<int32_t> free_list;   // front = next page handed out
  std::vector<uint8_t> in_use;     // per page id
};

struct dcpmla_reqmap {
  dcpmla_alloc* alloc = nullptr;
  int32_t max_requests = 0;
  int32_t max_pages = 0;
  std::vector<std::vector<int32_t>> pages;
  std::vector<int64_t> lens;
};

extern "C" {

const char* dcpmla_status_string(int status) {
  switch (status) {
    case DCPMLA_OK: return "ok";
    case DCPMLA_ERR_INVALID: return "invalid argument";
    case DCPMLA_ERR_UNSUPPORTED: return "unsupported dtype or shape";
    case DCPMLA_ERR_CAPACITY: return "capacity exhausted";
    case DCPMLA_ERR_CUDA: return "CUDA error";
    case DCPMLA_ERR_TIMEOUT: return "bounded device wait timed out";
    default: return "unknown status";
  }
}

int dcpmla_version(void) { return 1; }

int dcpmla_alloc_create(int32_t c, int64_t phys_capacity_tokens, int32_t phys_page,
                        const int32_t* initial_order, dcpmla_alloc** out) {
  if (!out) return DCPMLA_ERR_INVALID;
  *out = nullptr;
  if (c < 1 || c > DCPMLA_MAX_SHARDS || phys_page < 1 || phys_capacity_tokens < 0 ||
      phys_capacity_tokens % phys_page != 0)
    return DCPMLA_ERR_INVALID;
  const int64_t n = phys_capacity_tokens / phys_page;
  if (n > INT32_MAX) return DCPMLA_ERR_INVALID;
  // a virtual page id times the virtual page size must fit int64 slots
  if ((int64_t)phys_page * c > INT32_MAX) return DCPMLA_ERR_INVALID;
  dcpmla_alloc* a = new (std::nothrow) dcpmla_alloc();
  if (!a) return DCPMLA_ERR_CAPACITY;
  a->c = c;
  a->P = phys_page;
  a->num_pages = n;
  a->in_use.assign((size_t)n, 0);
  if (initial_order) {
    std::vector<uint8_t> seen((size_t)n, 0);
    for (int64_t i = 0; i < n; ++i) {
      const int32_t g = initial_order[i];
      if (g < 0 || g >= n || seen[(size_t)g]) {
        delete a;
        return DCPMLA_ERR_INVALID;
      }
      seen[(size_t)g] = 1;
      a->free_list.push_back(g);
    }
  } else {
    for (int64_t i = 0; i < n; ++i) a->free_list.push_back((int32_t)i);
  }
  *out = a;
  return DCPMLA_OK;
}

int dcpmla_alloc_destroy(dcpmla_alloc* a) {
  delete a;
  return DCPMLA_OK;
}

int dcpmla_alloc_geometry(const dcpmla_alloc* a, int32_t* c, int32_t* phys_page,
                          int32_t* virtual_page, int64_t* num_pages, int64_t* virtual_capacity) {
  if (!a) return DCPMLA_ERR_INVALID;
  if (c) *c = a->c;
  if (phys_page) *phys_page = a->P;
  if (virtual_page) *virtual_page = a->P * a->c;
  if (num_pages) *num_pages = a->num_pages;
  if (virtual_capacity) *virtual_capacity = a->num_pages * a->P * (int64_t)a->c;
  return DCPMLA_OK;
}

int dcpmla_effective_page_size(const dcpmla_alloc* a, int32_t* out) {
  if (!a || !out) return DCPMLA_ERR_INVALID;
  *out = a->P * a->c;
  return DCPMLA_OK;
}

int dcpmla_alloc_free_count(const dcpmla_alloc* a, int64_t* out) {
  if (!a || !out) return DCPMLA_ERR_INVALID;
  *out = (int64_t)a->free_list.size();
  return DCPMLA_OK;
}

int dcpmla_alloc_pages(dcpmla_alloc* a, int32_t n, int32_t* out_ids) {
  if (!a || n < 0 || (n > 0 && !out_ids)) return DCPMLA_ERR_INVALID;
  if ((size_t)n > a->free_list.size()) return DCPMLA_ERR_CAPACITY;
  for (int32_t i = 0; i < n; ++i) {
    const int32_t g = a->free_list.front();
    a->free_list.pop_front();
    a->in_use[(size_t)g] = 1;
    out_ids[i] = g;
  }
  return DCPMLA_OK;
}

int dcpmla_free_pages(dcpmla_alloc* a, int32_t n, const int32_t* ids) {
  if (!a || n < 0 || (n > 0 && !ids)) return DCPMLA_ERR_INVALID;
  // validate everything first: all-or-nothing
  std::vector<int32_t> sorted(ids, ids + n);
  std::sort(sorted.begin(), sorted.end());
  for (int32_t i = 0; i < n; ++i) {
    const int32_t g = sorted[(size_t)i];
    if (g < 0 || g >= a->num_pages || !a->in_use[(size_t)g]) return DCPMLA_ERR_INVALID;
    if (i > 0 && sorted[(size_t)i - 1] == g) return DCPMLA_ERR_INVALID;   // freed twice
  }
  for (int32_t i = 0; i < n; ++i) {
    a->in_use[(size_t)ids[i]] = 0;
    a->free_list.push_back(ids[i]);
  }
  return DCPMLA_OK;
}

int dcpmla_reqmap_create(dcpmla_alloc* a, int32_t max_requests, int32_t max_pages_per_request,
                         dcpmla_reqmap** out) {
  if (!out) return DCPMLA_ERR_INVALID;
  *out = nullptr;
  if (!a || max_requests < 1 || max_pages_per_request < 1) return DCPMLA_ERR_INVALID;
  dcpmla_reqmap* m = new (std::nothrow) dcpmla_reqmap();
  if (!m) return DCPMLA_ERR_CAPACITY;
  m->alloc = a;
  m->max_requests = max_requests;
  m->max_pages = max_pages_per_request;
  m->pages.resize((size_t)max_requests);
  m->lens.assign((size_t)max_requests, 0);
  *out = m;
  return DCPMLA_OK;
}

int dcpmla_reqmap_destroy(dcpmla_reqmap* m) {
  delete m;
  return DCPMLA_OK;
}

int dcpmla_reqmap_extend(dcpmla_reqmap* m, int32_t req, int64_t n_new,
                         int64_t* out_first_position) {
  if (!m || req < 0 || req >= m->max_requests || n_new < 0) return DCPMLA_ERR_INVALID;
  const int64_t vp = (int64_t)m->alloc->P * m->alloc->c;
  const int64_t cur = m->lens[(size_t)req];
  const int64_t want_len = cur + n_new;
  const int64_t want_pages = (want_len + vp - 1) / vp;
  std::vector<int32_t>& pg = m->pages[(size_t)req];
  const int64_t need = want_pages - (int64_t)pg.size();
  if (want_pages > m->max_pages) return DCPMLA_ERR_CAPACITY;
  if (need > 0) {
    std::vector<int32_t> ids((size_t)need);
    const int st = dcpmla_alloc_pages(m->alloc, (int32_t)need, ids.data());
    if (st != DCPMLA_OK) return st;
    pg.insert(pg.end(), ids.begin(), ids.end());
  }
  m->lens[(size_t)req] = want_len;
  if (out_first_position) *out_first_position = cur;
  return DCPMLA_OK;
}

int dcpmla_reqmap_release(dcpmla_reqmap* m, int32_t req) {
  if (!m || req < 0 || req >= m->max_requests) return DCPMLA_ERR_INVALID;
  std::vector<int32_t>& pg = m->pages[(size_t)req];
  const int st = dcpmla_free_pages(m->alloc, (int32_t)pg.size(), pg.data());
  if (st != DCPMLA_OK) return st;
  pg.clear();
  m->lens[(size_t)req] = 0;
  return DCPMLA_OK;
}

int dcpmla_reqmap_length(const dcpmla_reqmap* m, int32_t req, int64_t* out) {
  if (!m || !out || req < 0 || req >= m->max_requests) return DCPMLA_ERR_INVALID;
  *out = m->lens[(size_t)req];
  return DCPMLA_OK;
}

int dcpmla_reqmap_page_table(const dcpmla_reqmap* m, const int32_t* reqs, int32_t n_reqs,
                             int32_t max_pages, int32_t pad, int32_t* out_table,
                             int32_t* out_seq_lens) {
  if (!m || n_reqs < 0 || max_pages < 1 || (n_reqs > 0 && (!reqs || !out_table)))
    return DCPMLA_ERR_INVALID;
  for (int32_t i = 0; i < n_reqs; ++i) {
    const int32_t b = reqs[i];
    if (b < 0 || b >= m->max_requests) return DCPMLA_ERR_INVALID;
    if ((int64_t)m->pages[(size_t)b].size() > max_pages) return DCPMLA_ERR_CAPACITY;
    if (m->lens[(size_t)b] > INT32_MAX) return DCPMLA_ERR_UNSUPPORTED;
  }
  for (int32_t i = 0; i < n_reqs; ++i) {
    const std::vector<int32_t>& pg = m->pages[(size_t)reqs[i]];
    int32_t* row = out_table + (size_t)i * max_pages;
    for (int32_t k = 0; k < max_pages; ++k) row[k] = k < (int32_t)pg.size() ? pg[(size_t)k] : pad;
    if (out_seq_lens) out_seq_lens[i] = (int32_t)m->lens[(size_t)reqs[i]];
  }
  return DCPMLA_OK;
}

int dcpmla_map_positions(const int32_t* page_table, int32_t max_pages, int32_t c, int32_t interleave,
                         int32_t P, const int32_t* req, const int64_t* pos, int64_t n, int64_t* vslot,
                         int32_t* owner, int64_t* phys) {
  if (n < 0 || c < 1 || P < 1 || max_pages < 1) return DCPMLA_ERR_INVALID;
  if (interleave < 1 || P % interleave) return DCPMLA_ERR_INVALID;
  const int64_t I = interleave;
  if (n > 0 && (!page_table || !req || !pos)) return DCPMLA_ERR_INVALID;
  const int64_t vp = (int64_t)P * c;
  for (int64_t i = 0; i < n; ++i) {
    if (req[i] < 0 || pos[i] < 0) return DCPMLA_ERR_INVALID;
    const int64_t k = pos[i] / vp;
    if (k >= max_pages) return DCPMLA_ERR_INVALID;
    const int32_t g = page_table[(size_t)req[i] * max_pages + k];
    if (g < 0) return DCPMLA_ERR_INVALID;
    const int64_t v = (int64_t)g * vp + pos[i] % vp;
    if (vslot) vslot[i] = v;
    if (owner) owner[i] = (int32_t)((v / I) % c);
    if (phys) phys[i] = (v / (I * c)) * I + v % I;
  }
  return DCPMLA_OK;
}

}  // extern "C"
