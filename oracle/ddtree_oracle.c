/*
 * ddtree_oracle.c -- plain, slow, fp64 CPU oracle for DDTree verify attention
 * over an MLA latent KV pool.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's
 * CPU-baseline leg load this file's library.  It shares no code, header, table
 * or helper with the CUDA library; it follows the plain definition below and
 * nothing else (no tiling, no online softmax, no split of the key range).
 *
 * What is computed, for request b, tree node t, head h:
 *
 *   visible keys V(b,t) = { prefix positions j < L_b }  U  { tree nodes u : u == t
 *                          or u is an ancestor of t }
 *     - every draft node sees the whole shared prefix with no causal limit
 *       among the queries ("The Architecture Detective: Uncovering FlashMLA's
 *       Potential for Blackwell DDTree Verification", sections "The Message in
 *       Full" and "Assumptions and Their Validity");
 *     - among the tree nodes a node sees only its ancestors ("The Art of
 *       Systematic Investigation", section "Input Knowledge Required to
 *       Understand This Message", item 1) and itself.
 *   key/value row of prefix position j: pool[slot_idx[b][j]]; of tree node u:
 *     pool[tree_slot_idx[b][u]]  (page_size=1 token-slot table,
 *     "The Architecture Detective", section "The Message in Full").
 *   k = row[0:576] (512 latent + 64 rope), v = row[0:512] (one 576-wide latent
 *     row per slot, num_heads_k = 1; reading: v is the latent part).
 *   s_j   = sm_scale * sum_d q[b,t,h,d] * k_j[d]                (fp64)
 *   lse   = ln sum_{j in V} exp(s_j)                            (natural log)
 *   out_e = sum_{j in V} exp(s_j - lse) * v_j[e]
 *
 * Readings where the pages are silent:
 *   - nodes come in topological order: parent[0] = -1, parent[i] in [0, i);
 *     a parent entry outside that range is ignored (the node keeps itself and
 *     the prefix) and reported with status bit ORACLE_BAD_PARENT;
 *   - a slot index outside [0, pool_slots) removes that key from V and is
 *     reported with status bit ORACLE_BAD_SLOT.
 *
 * The mask is materialised in full: one byte per (node, key) of the request.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_BAD_SLOT 1
#define ORACLE_BAD_PARENT 2
#define ORACLE_BAD_ARGS 4

static double bf16_value(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/*
 * Tree part of the visibility mask of one request: vis[t*T + u] = 1 iff node u
 * is node t or one of its ancestors.  Returns status bits.
 */
int oracle_tree_visibility(const int32_t* parent, int T, uint8_t* vis) {
  int status = 0;
  memset(vis, 0, (size_t)T * (size_t)T);
  for (int t = 0; t < T; ++t) {
    int u = t;
    while (u >= 0) {
      vis[(size_t)t * T + u] = 1;
      int p = parent[u];
      int ok = (u == 0) ? (p == -1) : (p >= 0 && p < u);
      if (!ok) {
        status |= ORACLE_BAD_PARENT;
        break;
      }
      u = p;
    }
  }
  return status;
}

/*
 * Full mask of request b: mask[t*(L+T) + j], j < L prefix keys, j = L+u tree node u.
 * A key whose slot is out of range is masked out.
 */
static int build_mask(const int32_t* slot_row, int L, const int32_t* parent, const int32_t* tree_slot,
                      int T, int64_t pool_slots, uint8_t* mask) {
  int status = 0;
  int n = L + T;
  uint8_t* vis = (uint8_t*)malloc((size_t)T * (size_t)T);
  if (!vis) return ORACLE_BAD_ARGS;
  status |= oracle_tree_visibility(parent, T, vis);
  for (int t = 0; t < T; ++t) {
    uint8_t* m = mask + (size_t)t * n;
    for (int j = 0; j < L; ++j) m[j] = 1;
    for (int u = 0; u < T; ++u) m[L + u] = vis[(size_t)t * T + u];
  }
  for (int j = 0; j < L; ++j) {
    if (slot_row[j] < 0 || (int64_t)slot_row[j] >= pool_slots) {
      status |= ORACLE_BAD_SLOT;
      for (int t = 0; t < T; ++t) mask[(size_t)t * n + j] = 0;
    }
  }
  for (int u = 0; u < T; ++u) {
    if (tree_slot[u] < 0 || (int64_t)tree_slot[u] >= pool_slots) {
      status |= ORACLE_BAD_SLOT;
      for (int t = 0; t < T; ++t) mask[(size_t)t * n + L + u] = 0;
    }
  }
  free(vis);
  return status;
}

/*
 * Verify attention for the rows listed in `rows` (row id = (b*T + t)*H + h), or
 * for every row when rows == NULL.  out is [n_rows][d_v] fp64, lse is [n_rows].
 * A row with no visible key (only possible with bad slots) gets lse = -inf and
 * out = 0.  Returns the OR of the status bits of the requests touched.
 */
int oracle_verify_attn(const uint16_t* q, const uint16_t* pool, int64_t pool_slots,
                       const int32_t* slot_idx, int64_t slot_stride, const int32_t* prefix_len,
                       const int32_t* tree_parent, const int32_t* tree_slot_idx, int B, int T, int H,
                       int d_qk, int d_v, double sm_scale, const int64_t* rows, int64_t n_rows,
                       double* out, double* lse) {
  if (B < 0 || T < 1 || H < 1 || d_v > d_qk || d_v < 1) return ORACLE_BAD_ARGS;
  int64_t total = (int64_t)B * T * H;
  if (!rows) n_rows = total;
  int status = 0;

  /* materialise every request's mask */
  uint8_t** masks = (uint8_t**)calloc((size_t)(B > 0 ? B : 1), sizeof(uint8_t*));
  for (int b = 0; b < B; ++b) {
    int L = prefix_len[b];
    if (L < 0 || L > slot_stride) { status |= ORACLE_BAD_ARGS; L = 0; }
    masks[b] = (uint8_t*)malloc((size_t)T * (size_t)(L + T));
    status |= build_mask(slot_idx + (int64_t)b * slot_stride, L, tree_parent + (int64_t)b * T,
                         tree_slot_idx + (int64_t)b * T, T, pool_slots, masks[b]);
  }
  if (status & ORACLE_BAD_ARGS) {
    for (int b = 0; b < B; ++b) free(masks[b]);
    free(masks);
    return status;
  }

#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t i = 0; i < n_rows; ++i) {
    int64_t row = rows ? rows[i] : i;
    int b = (int)(row / ((int64_t)T * H));
    int t = (int)((row / H) % T);
    int L = prefix_len[b];
    int n = L + T;
    const uint8_t* m = masks[b] + (size_t)t * n;
    const uint16_t* qrow = q + row * d_qk;
    double* o = out + i * d_v;
    double* s = (double*)malloc(sizeof(double) * (size_t)n);
    const uint16_t** kv = (const uint16_t**)malloc(sizeof(uint16_t*) * (size_t)n);

    /* scores of the visible keys */
    double smax = -INFINITY;
    for (int j = 0; j < n; ++j) {
      if (!m[j]) continue;
      int64_t slot = (j < L) ? slot_idx[(int64_t)b * slot_stride + j]
                             : tree_slot_idx[(int64_t)b * T + (j - L)];
      kv[j] = pool + slot * d_qk;
      double dot = 0.0;
      for (int d = 0; d < d_qk; ++d) dot += bf16_value(qrow[d]) * bf16_value(kv[j][d]);
      s[j] = sm_scale * dot;
      if (s[j] > smax) smax = s[j];
    }

    for (int e = 0; e < d_v; ++e) o[e] = 0.0;
    if (smax == -INFINITY) {
      lse[i] = -INFINITY;
    } else {
      double z = 0.0;
      for (int j = 0; j < n; ++j)
        if (m[j]) z += exp(s[j] - smax);
      double l = smax + log(z);
      lse[i] = l;
      for (int j = 0; j < n; ++j) {
        if (!m[j]) continue;
        double p = exp(s[j] - l);
        for (int e = 0; e < d_v; ++e) o[e] += p * bf16_value(kv[j][e]);
      }
    }
    free(kv);
    free(s);
  }

  for (int b = 0; b < B; ++b) free(masks[b]);
  free(masks);
  return status;
}

/*
 * kv_compact: copy request b's prefix rows to consecutive destination slots
 * dst_start[b] + j and return the rewritten slot table.  Plain row copies.
 */
int oracle_kv_compact(const uint16_t* src, uint16_t* dst, int64_t pool_slots, const int32_t* slot_idx,
                      int64_t slot_stride, const int32_t* prefix_len, const int64_t* dst_start, int B,
                      int d_qk, int32_t* slot_idx_out) {
  int status = 0;
  for (int b = 0; b < B; ++b) {
    for (int j = 0; j < prefix_len[b]; ++j) {
      int64_t from = slot_idx[(int64_t)b * slot_stride + j];
      int64_t to = dst_start[b] + j;
      if (from < 0 || from >= pool_slots || to < 0 || to >= pool_slots) {
        status |= ORACLE_BAD_SLOT;
        continue;
      }
      memcpy(dst + to * d_qk, src + from * d_qk, sizeof(uint16_t) * (size_t)d_qk);
      slot_idx_out[(int64_t)b * slot_stride + j] = (int32_t)to;
    }
  }
  return status;
}

/*
 * Sparse-index variant ("The Architecture Detective: Uncovering FlashMLA's
 * Potential for Blackwell DDTree Verification", sections "The Message in Full"
 * and "The Discovery: FlashMLA's Hidden Capabilities": a sparse attention call
 * takes, per query, a fixed-length list of key indices in which -1 marks an
 * invalid entry).  Here every query node lists its own keys: node (b, t) owns
 * indices[(b*T + t)*topk .. +topk); all H heads of the node attend to the rows
 * pool[slot] for the listed slots != -1.  A slot listed twice counts twice.
 * A listed value outside [0, pool_slots) other than -1 is left out and
 * reported with ORACLE_BAD_SLOT.  A node with no key gets lse = -inf, out = 0.
 *   s_i   = sm_scale * q . pool[slot_i][0:d_qk]               (fp64)
 *   lse   = ln sum_i exp(s_i),  out_e = sum_i exp(s_i - lse) * pool[slot_i][e]
 */
int oracle_verify_sparse(const uint16_t* q, const uint16_t* pool, int64_t pool_slots, const int32_t* indices,
                         int topk, int B, int T, int H, int d_qk, int d_v, double sm_scale, double* out,
                         double* lse) {
  if (B < 0 || T < 1 || H < 1 || topk < 0 || d_v > d_qk || d_v < 1) return ORACLE_BAD_ARGS;
  int flags = 0;
  for (int64_t i = 0; i < (int64_t)B * T * topk; ++i)
    if (indices[i] != -1 && (indices[i] < 0 || (int64_t)indices[i] >= pool_slots)) flags |= ORACLE_BAD_SLOT;
  const int64_t n_rows = (int64_t)B * T * H;

#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t row = 0; row < n_rows; ++row) {
    const int32_t* list = indices + (row / H) * topk;
    const uint16_t* query = q + row * (int64_t)d_qk;
    double* score = (double*)malloc(sizeof(double) * (size_t)(topk > 0 ? topk : 1));
    unsigned char* listed = (unsigned char*)malloc((size_t)(topk > 0 ? topk : 1));
    double best = -INFINITY;
    for (int k = 0; k < topk; ++k) {
      const int64_t slot = list[k];
      listed[k] = slot >= 0 && slot < pool_slots;
      if (!listed[k]) continue;
      const uint16_t* key = pool + slot * d_qk;
      double acc = 0.0;
      for (int c = 0; c < d_qk; ++c) acc += bf16_value(query[c]) * bf16_value(key[c]);
      score[k] = sm_scale * acc;
      if (score[k] > best) best = score[k];
    }
    double* orow = out + row * (int64_t)d_v;
    for (int c = 0; c < d_v; ++c) orow[c] = 0.0;
    if (best == -INFINITY) {
      lse[row] = -INFINITY;
    } else {
      double total = 0.0;
      for (int i = 0; i < topk; ++i)
        if (listed[i]) total += exp(score[i] - best);
      const double log_norm = best + log(total);
      lse[row] = log_norm;
      for (int n = 0; n < topk; ++n) {
        if (!listed[n]) continue;
        const double weight = exp(score[n] - log_norm);
        const uint16_t* val = pool + (int64_t)list[n] * d_qk;
        for (int c = 0; c < d_v; ++c) orow[c] += weight * bf16_value(val[c]);
      }
    }
    free(listed);
    free(score);
  }
  return flags;
}
