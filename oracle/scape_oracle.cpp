/*
 * SCAPE oracle: a plain, slow, single-threaded CPU statement of one SCAPE
 * optimizer step, written to be checked against the method's description by
 * eye.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's
 * CPU-baseline and reference legs may load this library; the product path
 * never does.  It shares no code, header or helper with the CUDA path.
 *
 * Source: "SCAPE: Accurate and Efficient LLM Training with Extreme Sparse
 * Communication" (arXiv 2607.01678): abstract; gist.science technical summary,
 * §2 "Methodology" (AdamS base optimizer, partitioned mask synchronization,
 * delayed mask usage, single-buffer second-moment reconstruction) and §3.
 * The pages give the method in prose only; the exact per-step rule this file
 * follows is:
 *
 *   (1) u_w = b1*u_w + (1-b1)*g_w                   per-worker first moment
 *   (2) a_w = e_w + u_w                             accumulator (error feedback)
 *   (3) b_w = a_w (.) M_{t-1}                       sparse buffer, delayed mask
 *   (4) e_w = a_w - b_w                             residual
 *   (5) bbar = (1/W) sum_w b_w, w = 0..W-1 in order the one synchronized buffer
 *   (6) v = b2*v + (1-b2)*bbar^2                    second moment from bbar
 *   (7) theta -= lr*(bbar/(sqrt(v)+eps) + wd*theta) AdamS update + weight decay
 *   (8) worker w owns shard w; in every chunk of its shard it keeps the top-k
 *       of |a_w|, ties going to the lower index
 *   (9) the shard masks, concatenated, are M_t; M_t is applied at step t+1.
 *
 * Readings where the pages leave a step open:
 *   - all arithmetic is IEEE fp32, round-to-nearest-even, evaluated with the
 *     parenthesisation written below and no fused multiply-add (build with
 *     -ffp-contract=off); bf16 gradients widen to fp32 exactly;
 *   - (1-b1), (1-b2) and 1/W are fp32 operations on the fp32 inputs;
 *   - "(.) M" is a select: off the mask b = +0 (so a = b + e holds exactly);
 *   - no bias correction (none is described);
 *   - the sum in (5) runs over the coordinates of M_{t-1} only; off the mask
 *     bbar = +0, and (6)-(7) still run there (v decays, theta decays);
 *   - top-k key: |a| as the fp32 bit pattern with the sign cleared, compared
 *     as an unsigned integer; k_c = floor(density * len_c) in IEEE double;
 *   - chunks of C coordinates tile the flat parameter vector, ignoring tensor
 *     boundaries (or, in the per-tensor variant, tile each tensor separately,
 *     the pages' "partitioned layers"); with n_ch chunks and q = ceil(n_ch/W),
 *     worker w owns chunks [w*q, min((w+1)*q, n_ch));
 *   - step 0 has no earlier mask: M_{-1} is the selection (8) applied to the
 *     step-0 accumulators a_w = e_w + (b1*u_w + (1-b1)*g_w) before anything
 *     is written, so every step carries exactly k_c coordinates per chunk.
 *
 * Domain: the per-coordinate rule (1)-(7) involves only coordinate i across
 * workers, and (8) involves only one chunk, so the oracle may run on any set
 * of whole chunks (the "domain") and give, for those chunks, exactly what a
 * run over all chunks gives.  Arrays below are indexed by domain position;
 * dom_index[] holds the flat coordinate of each position.
 */
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <new>
#include <vector>

#define OR_API extern "C" __attribute__((visibility("default")))

namespace {

struct Chunk {
  uint64_t start;   // flat index of the first coordinate
  uint32_t len;     // coordinates in the chunk
  uint32_t k;       // coordinates kept
  int owner;        // worker owning the chunk
  uint64_t dom0;    // domain position of the first coordinate
};

struct Oracle {
  // hyper-parameters and geometry
  uint64_t N = 0;
  uint32_t C = 0;
  int W = 0;
  double density = 0;
  float b1 = 0, b2 = 0, lr = 0, wd = 0, eps = 0;
  uint64_t n_chunks_total = 0;
  bool union_mask = false;            // the non-partitioned variant (union of W top-k)
  std::vector<Chunk> chunks;          // the domain's chunks, ascending
  std::vector<uint64_t> all_start, all_len, all_k;  // every chunk of the layout
  std::vector<uint64_t> dom_index;    // flat index of each domain position
  uint64_t n = 0;                     // domain size

  // optimizer state over the domain
  std::vector<float> theta, v;        // [n]
  std::vector<float> u, e;            // [W][n]
  std::vector<uint8_t> mask_prev;     // M_{t-1}: one byte per coordinate (0/1)
  long t = 0;

  // what the last step produced, kept for the tests
  std::vector<uint8_t> mask_used;     // the mask applied in the last step
  std::vector<float> a_last, b_last;  // [W][n] accumulators and sparse buffers
  std::vector<std::vector<float>> vals;  // [W] compact sparse buffers, ascending index
  std::vector<float> bbar;            // compact synchronized buffer
  std::vector<uint64_t> sel_index;    // flat index of each compact entry
};

float bf16_to_f32(uint16_t h) {
  uint32_t bits = (uint32_t)h << 16;
  float f;
  std::memcpy(&f, &bits, 4);
  return f;
}

uint32_t topk_key(float a) {
  uint32_t bits;
  std::memcpy(&bits, &a, 4);
  return bits & 0x7fffffffu;
}

// Step (8) on one chunk: keep the k largest keys, equal keys ordered by
// ascending index; writes 1 for kept, 0 otherwise.
void select_topk(const float* a, uint32_t len, uint32_t k, uint8_t* keep) {
  std::vector<uint32_t> order(len);
  for (uint32_t i = 0; i < len; i++) order[i] = i;
  std::sort(order.begin(), order.end(), [&](uint32_t x, uint32_t y) {
    uint32_t kx = topk_key(a[x]), ky = topk_key(a[y]);
    if (kx != ky) return kx > ky;
    return x < y;
  });
  for (uint32_t i = 0; i < len; i++) keep[i] = 0;
  for (uint32_t r = 0; r < k; r++) keep[order[r]] = 1;
}

// (8)-(9): build the mask of the whole domain from the owners' accumulators
// a[W][n]; the shard masks land side by side, which is the concatenation.
void partitioned_select(const Oracle& o, const std::vector<float>& a, std::vector<uint8_t>& mask) {
  for (const Chunk& c : o.chunks) {
    const float* aw = a.data() + (uint64_t)c.owner * o.n + c.dom0;
    select_topk(aw, c.len, c.k, mask.data() + c.dom0);
  }
}

// The non-partitioned alternative the pages set SCAPE against (technical
// summary §2, "Partitioned Mask Synchronization": without partitioning, each
// worker's own top-k lands on different coordinates and the synchronized set
// fills in): every worker ranks its own accumulator in every chunk with the
// same key and tie rule, and the mask is the union of the W selections.
void union_select(const Oracle& o, const std::vector<float>& a, std::vector<uint8_t>& mask) {
  std::vector<uint8_t> keep;
  for (const Chunk& c : o.chunks) {
    uint8_t* m = mask.data() + c.dom0;
    for (uint32_t i = 0; i < c.len; i++) m[i] = 0;
    keep.resize(c.len);
    for (int w = 0; w < o.W; w++) {
      select_topk(a.data() + (uint64_t)w * o.n + c.dom0, c.len, c.k, keep.data());
      for (uint32_t i = 0; i < c.len; i++) m[i] |= keep[i];
    }
  }
}

void select_mask(const Oracle& o, const std::vector<float>& a, std::vector<uint8_t>& mask) {
  if (o.union_mask) union_select(o, a, mask);
  else partitioned_select(o, a, mask);
}

void oracle_step_impl(Oracle& o, const uint16_t* grads /* [W][n] */) {
  const uint64_t n = o.n;
  const int W = o.W;
  const float c1 = 1.0f - o.b1;
  const float c2 = 1.0f - o.b2;
  const float invW = 1.0f / (float)W;

  if (o.t == 0) {
    // M_{-1}: selection on the step-0 accumulators, nothing written yet.
    std::vector<float> a0((uint64_t)W * n);
    for (int w = 0; w < W; w++)
      for (uint64_t i = 0; i < n; i++) {
        uint64_t x = (uint64_t)w * n + i;
        float g = bf16_to_f32(grads[x]);
        float un = (o.b1 * o.u[x]) + (c1 * g);
        a0[x] = o.e[x] + un;
      }
    select_mask(o, a0, o.mask_prev);
  }

  // (1)-(4) on every worker; the kept values are compacted in index order.
  o.mask_used = o.mask_prev;
  for (int w = 0; w < W; w++) {
    o.vals[w].clear();
    for (uint64_t i = 0; i < n; i++) {
      uint64_t x = (uint64_t)w * n + i;
      float g = bf16_to_f32(grads[x]);
      o.u[x] = (o.b1 * o.u[x]) + (c1 * g);                 // (1)
      float a = o.e[x] + o.u[x];                            // (2)
      float b = o.mask_prev[i] ? a : 0.0f;                  // (3)
      o.e[x] = a - b;                                       // (4)
      o.a_last[x] = a;
      o.b_last[x] = b;
      if (o.mask_prev[i]) o.vals[w].push_back(b);
    }
  }

  // (5): the synchronized buffer, summed over workers in order 0..W-1.
  o.sel_index.clear();
  for (uint64_t i = 0; i < n; i++)
    if (o.mask_prev[i]) o.sel_index.push_back(o.dom_index[i]);
  const uint64_t K = o.vals[0].size();
  o.bbar.assign(K, 0.0f);
  for (uint64_t p = 0; p < K; p++) {
    float s = o.vals[0][p];
    for (int w = 1; w < W; w++) s = s + o.vals[w][p];
    o.bbar[p] = s * invW;
  }

  // (6)-(7) on every coordinate; bbar is +0 off the mask.
  uint64_t p = 0;
  for (uint64_t i = 0; i < n; i++) {
    float bb = 0.0f;
    if (o.mask_prev[i]) bb = o.bbar[p++];
    o.v[i] = (o.b2 * o.v[i]) + (c2 * (bb * bb));                    // (6)
    float q = bb / (std::sqrt(o.v[i]) + o.eps);
    o.theta[i] = o.theta[i] - (o.lr * (q + (o.wd * o.theta[i])));   // (7)
  }

  // (8)-(9): next mask from the owners' accumulators (every worker's, in the
  // union variant); used at step t+1.
  select_mask(o, o.a_last, o.mask_prev);
  o.t += 1;
}

enum { OR_THETA = 0, OR_V = 1, OR_U = 2, OR_E = 3, OR_A = 4, OR_B = 5 };

}  // namespace

/* Create an oracle for the flat layout of n_tensors tensors (numel[]), chunk
 * size C, W workers.  chunk_ids[0..n_ids) (ascending, distinct) picks the
 * domain; n_ids == 0 means every chunk.  flags: 1 = chunks restart at every
 * tensor; 2 = the non-partitioned variant (the mask is the union of every
 * worker's own top-k in every chunk).  Returns nullptr on bad arguments. */
OR_API void* oracle_create(const uint64_t* numel, uint32_t n_tensors, uint32_t C, int W,
                           double density, float b1, float b2, float lr, float wd, float eps,
                           const uint64_t* chunk_ids, uint64_t n_ids, int flags) {
  const int per_tensor = flags & 1;
  if (!numel || n_tensors == 0 || C == 0 || W < 1 || !(density > 0.0 && density <= 1.0))
    return nullptr;
  Oracle* o = new (std::nothrow) Oracle();
  if (!o) return nullptr;
  for (uint32_t i = 0; i < n_tensors; i++) o->N += numel[i];
  if (o->N == 0) { delete o; return nullptr; }
  o->C = C; o->W = W; o->density = density;
  o->union_mask = (flags & 2) != 0;
  o->b1 = b1; o->b2 = b2; o->lr = lr; o->wd = wd; o->eps = eps;
  // Chunk boundaries: every C coordinates of the flat vector, or (per_tensor)
  // every C coordinates of each tensor, its last chunk shorter.
  std::vector<uint64_t> cstart;
  if (per_tensor) {
    uint64_t off = 0;
    for (uint32_t t = 0; t < n_tensors; t++) {
      for (uint64_t x = 0; x < numel[t]; x += C) cstart.push_back(off + x);
      off += numel[t];
    }
  } else {
    for (uint64_t x = 0; x < o->N; x += C) cstart.push_back(x);
  }
  o->n_chunks_total = cstart.size();
  for (size_t c = 0; c < cstart.size(); c++) {
    const uint64_t end = c + 1 < cstart.size() ? cstart[c + 1] : o->N;
    o->all_start.push_back(cstart[c]);
    o->all_len.push_back(end - cstart[c]);
    o->all_k.push_back((uint64_t)std::floor(density * (double)(end - cstart[c])));
  }
  const uint64_t q = (o->n_chunks_total + W - 1) / W;
  std::vector<uint64_t> ids;
  if (n_ids == 0) {
    for (uint64_t c = 0; c < o->n_chunks_total; c++) ids.push_back(c);
  } else {
    for (uint64_t j = 0; j < n_ids; j++) {
      if (chunk_ids[j] >= o->n_chunks_total || (j > 0 && chunk_ids[j] <= chunk_ids[j - 1])) {
        delete o;
        return nullptr;
      }
      ids.push_back(chunk_ids[j]);
    }
  }
  for (uint64_t c : ids) {
    Chunk ch;
    ch.start = cstart[c];
    uint64_t end = c + 1 < cstart.size() ? cstart[c + 1] : o->N;
    ch.len = (uint32_t)(end - ch.start);
    ch.k = (uint32_t)std::floor(density * (double)ch.len);
    ch.owner = (int)(c / q);
    ch.dom0 = o->n;
    for (uint64_t i = ch.start; i < end; i++) o->dom_index.push_back(i);
    o->n += ch.len;
    o->chunks.push_back(ch);
  }
  o->theta.assign(o->n, 0.0f);
  o->v.assign(o->n, 0.0f);
  o->u.assign((uint64_t)W * o->n, 0.0f);
  o->e.assign((uint64_t)W * o->n, 0.0f);
  o->a_last.assign((uint64_t)W * o->n, 0.0f);
  o->b_last.assign((uint64_t)W * o->n, 0.0f);
  o->mask_prev.assign(o->n, 0);
  o->mask_used.assign(o->n, 0);
  o->vals.assign(W, {});
  return o;
}

OR_API void oracle_destroy(void* h) { delete static_cast<Oracle*>(h); }

OR_API uint64_t oracle_domain_size(void* h) { return static_cast<Oracle*>(h)->n; }
OR_API long oracle_step_count(void* h) { return static_cast<Oracle*>(h)->t; }

/* Flat indices of the domain positions. */
OR_API void oracle_domain_index(void* h, uint64_t* out) {
  Oracle* o = static_cast<Oracle*>(h);
  std::memcpy(out, o->dom_index.data(), o->n * sizeof(uint64_t));
}

/* Per domain chunk: start, len, k, owner. */
OR_API uint64_t oracle_chunks(void* h, uint64_t* start, uint32_t* len, uint32_t* k, int32_t* owner) {
  Oracle* o = static_cast<Oracle*>(h);
  for (size_t j = 0; j < o->chunks.size(); j++) {
    if (start) start[j] = o->chunks[j].start;
    if (len) len[j] = o->chunks[j].len;
    if (k) k[j] = o->chunks[j].k;
    if (owner) owner[j] = o->chunks[j].owner;
  }
  return o->chunks.size();
}

/* Every chunk of the layout (not only the domain): start, len, k. Returns the
 * chunk count; any pointer may be NULL. */
OR_API uint64_t oracle_all_chunks(void* h, uint64_t* start, uint64_t* len, uint64_t* k) {
  Oracle* o = static_cast<Oracle*>(h);
  for (size_t j = 0; j < o->all_start.size(); j++) {
    if (start) start[j] = o->all_start[j];
    if (len) len[j] = o->all_len[j];
    if (k) k[j] = o->all_k[j];
  }
  return o->all_start.size();
}

/* One step; grads[W][n] are bf16 bit patterns over the domain. */
OR_API int oracle_step(void* h, const uint16_t* grads) {
  if (!h || !grads) return -1;
  oracle_step_impl(*static_cast<Oracle*>(h), grads);
  return 0;
}

static std::vector<float>* field_of(Oracle* o, int which) {
  switch (which) {
    case OR_THETA: return &o->theta;
    case OR_V: return &o->v;
    case OR_U: return &o->u;
    case OR_E: return &o->e;
    case OR_A: return &o->a_last;
    case OR_B: return &o->b_last;
    default: return nullptr;
  }
}

/* Read a float field over the domain: THETA/V ignore w; U/E/A/B take worker w. */
OR_API int oracle_get(void* h, int which, int w, float* out) {
  Oracle* o = static_cast<Oracle*>(h);
  std::vector<float>* f = field_of(o, which);
  if (!f) return -1;
  uint64_t off = 0;
  if (which >= OR_U) {
    if (w < 0 || w >= o->W) return -1;
    off = (uint64_t)w * o->n;
  }
  std::memcpy(out, f->data() + off, o->n * sizeof(float));
  return 0;
}

/* Overwrite a float field (THETA, V, U, E) over the domain. */
OR_API int oracle_set(void* h, int which, int w, const float* src) {
  Oracle* o = static_cast<Oracle*>(h);
  if (which > OR_E) return -1;
  std::vector<float>* f = field_of(o, which);
  uint64_t off = 0;
  if (which >= OR_U) {
    if (w < 0 || w >= o->W) return -1;
    off = (uint64_t)w * o->n;
  }
  std::memcpy(f->data() + off, src, o->n * sizeof(float));
  return 0;
}

/* Masks, one byte per domain position: which 0 = mask generated by the last
 * step (applied at the next one), 1 = mask applied in the last step. */
OR_API int oracle_get_mask(void* h, int which, uint8_t* out) {
  Oracle* o = static_cast<Oracle*>(h);
  const std::vector<uint8_t>& m = which == 0 ? o->mask_prev : o->mask_used;
  std::memcpy(out, m.data(), o->n);
  return 0;
}

/* Set the mask to apply at the next step and the step counter (resume). */
OR_API int oracle_set_mask(void* h, const uint8_t* src, long t) {
  Oracle* o = static_cast<Oracle*>(h);
  for (uint64_t i = 0; i < o->n; i++) o->mask_prev[i] = src[i] ? 1 : 0;
  o->t = t;
  return 0;
}

/* Compact buffers of the last step: w in [0, W) -> worker w's kept values,
 * w == -1 -> the synchronized buffer bbar, w == -2 -> flat indices (as
 * float-free uint64 in idx).  Returns the entry count. */
OR_API uint64_t oracle_get_sparse(void* h, int w, float* vals, uint64_t* idx) {
  Oracle* o = static_cast<Oracle*>(h);
  const std::vector<float>* src = nullptr;
  if (w == -1) src = &o->bbar;
  else if (w >= 0 && w < o->W) src = &o->vals[w];
  uint64_t cnt = o->sel_index.size();
  if (vals && src) std::memcpy(vals, src->data(), cnt * sizeof(float));
  if (idx) std::memcpy(idx, o->sel_index.data(), cnt * sizeof(uint64_t));
  return cnt;
}

/* Step (8) alone on one array: keep[i] = 1 for the k kept coordinates. */
OR_API int oracle_topk(const float* a, uint32_t len, uint32_t k, uint8_t* keep) {
  if (!a || !keep || k > len) return -1;
  select_topk(a, len, k, keep);
  return 0;
}

/* Dense AdamS under data parallelism, the comparator the SCAPE pages measure
 * against (abstract: "3.26x speedup per step compared to dense AdamS";
 * gist.science technical summary §4).  Every worker's full gradient is
 * averaged (the dense all-reduce, workers summed in order 0..W-1), then one
 * AdamS update, whose second moment is the EMA of the squared momentum:
 *   gbar  = (g_0 + ... + g_{W-1}) * (1/W)
 *   m     = b1*m + (1-b1)*gbar
 *   v     = b2*v + (1-b2)*(m*m)
 *   theta = theta - lr*(m/(sqrt(v)+eps) + wd*theta)
 * fp32 with the same conventions as the SCAPE step above.  grads[W][n]. */
OR_API int oracle_dense_adams_step(float* theta, float* m, float* v, const uint16_t* grads,
                                   uint64_t n, int W, float b1, float b2, float lr, float wd,
                                   float eps) {
  if (!theta || !m || !v || !grads || W < 1) return -1;
  const float c1 = 1.0f - b1;
  const float c2 = 1.0f - b2;
  const float invW = 1.0f / (float)W;
  for (uint64_t i = 0; i < n; i++) {
    float s = bf16_to_f32(grads[i]);
    for (int w = 1; w < W; w++) s = s + bf16_to_f32(grads[(uint64_t)w * n + i]);
    const float gbar = s * invW;
    m[i] = (b1 * m[i]) + (c1 * gbar);
    v[i] = (b2 * v[i]) + (c2 * (m[i] * m[i]));
    const float q = m[i] / (std::sqrt(v[i]) + eps);
    theta[i] = theta[i] - (lr * (q + (wd * theta[i])));
  }
  return 0;
}
