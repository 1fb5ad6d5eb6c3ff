// Workspace layout and argument checks shared by the entry points and the
// kernel launchers (host code).
#pragma once
#include <stddef.h>
#include <stdint.h>

#include <algorithm>
#include <vector>

#include "../../include/sage.h"

namespace sage {

inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

constexpr int kMaxTokens = 1 << 23;  // fixed-point means stay exact in int64 up to here

// Statistics scratch of the quantize pre-pass, per (b, kv-head) and channel:
// K column sums and V column sums as fixed-point int64 (lsb 2^-24), V column
// min and max as order-preserving int32 encodings of the fp32 values.
struct StatsView {
  int64_t *ksum;  // [B*Hkv, d]
  int64_t *vsum;  // [B*Hkv, d]
  int *vmin;      // [B*Hkv, d]
  int *vmax;      // [B*Hkv, d]
};

inline size_t stats_bytes(const sage_shape &s) {
  const size_t n = (size_t)s.B * s.Hkv * s.d;
  return n * (8 + 8 + 4 + 4);
}

// Argument checks common to every entry point.  Returns SAGE_OK or the reason.
inline sage_status check_request(const sage_shape *s, int mode, int bq, int bk) {
  if (!s) return SAGE_ERR_INVALID_ARG;
  if (s->B <= 0 || s->Hq <= 0 || s->Hkv <= 0 || s->N <= 0 || s->M <= 0 || s->d <= 0)
    return SAGE_ERR_INVALID_ARG;
  if (s->Hq % s->Hkv != 0) return SAGE_ERR_INVALID_ARG;
  if (mode < SAGE_Q8_PV8 || mode > SAGE_SAGEBWD_I8) return SAGE_ERR_INVALID_ARG;
  if (bq <= 0 || bk <= 0) return SAGE_ERR_INVALID_ARG;
  if (s->N > kMaxTokens || s->M > kMaxTokens) return SAGE_ERR_UNSUPPORTED;
  if (s->d != 64 && s->d != 128) return SAGE_ERR_UNSUPPORTED;
  if (bq != 128) return SAGE_ERR_UNSUPPORTED;
  if (bk != 64 && bk != 128) return SAGE_ERR_UNSUPPORTED;
  // SageBwd: 16-bit P^ and V^ tiles fit the shared memory with 64-key tiles
  if (mode == SAGE_SAGEBWD_I8 && bk != 64) return SAGE_ERR_UNSUPPORTED;
  if ((int64_t)s->B * s->Hq > (1 << 20) || (int64_t)s->B * s->Hkv > (1 << 20)) return SAGE_ERR_UNSUPPORTED;
  return SAGE_OK;
}

inline sage_status compute_layout(const sage_shape *s, int mode, int bq, int bk, sage_ws_layout *L) {
  sage_status st = check_request(s, mode, bq, bk);
  if (st != SAGE_OK) return st;
  const int64_t B = s->B, Hq = s->Hq, Hkv = s->Hkv, d = s->d;
  const int64_t N_pad = align_up((size_t)s->N, 128), M_pad = align_up((size_t)s->M, 128);
  const int64_t Tm = N_pad / bq, Tn = cdiv(s->M, bk);
  // bytes per stored code: fp16 integer (modes 0, 3), E4M3 byte (1), packed E2M1 (2)
  const bool i8 = (mode == SAGE_Q8_PV8 || mode == SAGE_SAGEBWD_I8);
  const double code_bytes = i8 ? 2.0 : (mode == SAGE_QF8_PV8 ? 1.0 : 0.5);
  const double v_bytes = (mode == SAGE_NVFP4) ? 0.5 : (mode == SAGE_SAGEBWD_I8 ? 2.0 : 1.0);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align_up(off + (bytes ? bytes : 1), 1024);
    return o;
  };
  L->qhat = take((size_t)(B * Hq * N_pad * d * code_bytes));
  L->dq = take((size_t)(B * Hq * Tm * 4));
  L->qbar = take((size_t)(B * Hq * Tm * d * 4));
  L->khat = take((size_t)(B * Hkv * M_pad * d * code_bytes));
  L->dk = take((size_t)(B * Hkv * Tn * 4));
  L->kbar = take((size_t)(B * Hkv * d * 4));
  L->vhat = take((size_t)(B * Hkv * d * M_pad * v_bytes));
  L->dv = take((size_t)(B * Hkv * d * 4));
  L->vm = take((size_t)(B * Hkv * d * 4));
  // NVFP4 block scales: one E4M3 byte per 16 codes
  const bool fp4 = (mode == SAGE_NVFP4);
  L->qsf = take(fp4 ? (size_t)(B * Hq * N_pad * (d / 16)) : 0);
  L->ksf = take(fp4 ? (size_t)(B * Hkv * M_pad * (d / 16)) : 0);
  // V scales: per (b, kv-head) ceil(d/128) atoms of 128 channel rows, each
  // holding M_pad/16 token blocks
  L->vsf = take(fp4 ? (size_t)(B * Hkv * cdiv(d, 128) * 128 * (M_pad / 16)) : 0);
  L->stats = take(stats_bytes(*s));
  L->status = take(16);
  L->dqt = take((size_t)(B * Hq * N_pad * 4));
  L->dvb = take(mode == SAGE_SAGEBWD_I8 ? (size_t)(B * Hkv * Tn * 4) : 0);
  L->lse = take(mode == SAGE_SAGEBWD_I8 ? (size_t)(B * Hq * N_pad * 4) : 0);
  // the backward's inputs (sage_bwd_prepare)
  L->doc = take(mode == SAGE_SAGEBWD_I8 ? (size_t)(B * Hq * N_pad * d * 2) : 0);
  L->dos = take(mode == SAGE_SAGEBWD_I8 ? (size_t)(B * Hq * Tm * 4) : 0);
  L->drow = take(mode == SAGE_SAGEBWD_I8 ? (size_t)(B * Hq * N_pad * 4) : 0);
  L->total = off;
  L->N_pad = (int)N_pad;
  L->M_pad = (int)M_pad;
  L->Tm = (int)Tm;
  L->Tn = (int)Tn;
  return SAGE_OK;
}

// ------------------------------------------------------------------ packed sequences
// A packed-sequence request runs on the batched workspace layout with B = the
// number of sequences, N = the longest query run and M = the longest key run:
// sequence b's codes sit where batch b's would, so every tensor map and
// workspace index stays as in the batched case, and each kernel takes the
// sequence's own lengths from this table.  q0 / k0: the sequence's first row
// in the packed [total, H, d] inputs.
struct VarSeq {
  int N, M, q0, k0;
};

struct VarlenPlan {
  sage_shape shape;     // B = nseq, N = max query run, M = max key run
  sage_ws_layout L;     // the batched layout of that shape
  size_t seq_off;       // VarSeq[nseq], after the batched regions
  size_t item_off;      // int[items]: work item codes bh * Tm + qi
  size_t total;         // workspace bytes
  int items;            // work items (query blocks of non-empty sequences)
  std::vector<VarSeq> seqs;
  std::vector<int> item_codes;
};

// Checks cu_seqlens (host, nseq + 1 entries each, starting at 0, non-decreasing,
// every run within the token limit; a sequence with queries needs keys, and
// under a causal mask at least as many keys as queries) and builds the plan:
// work items longest first (most key tiles), as in the batched kernels.
inline sage_status plan_varlen(int nseq, const int *cu_q, const int *cu_k, int Hq, int Hkv, int d, int mode,
                               int bq, int bk, int causal, VarlenPlan *P) {
  if (nseq <= 0 || !cu_q || !cu_k || !P) return SAGE_ERR_INVALID_ARG;
  if (cu_q[0] != 0 || cu_k[0] != 0) return SAGE_ERR_INVALID_ARG;
  int max_q = 0, max_k = 0;
  P->seqs.assign((size_t)nseq, VarSeq{0, 0, 0, 0});
  for (int b = 0; b < nseq; ++b) {
    const long long nq = (long long)cu_q[b + 1] - cu_q[b], nk = (long long)cu_k[b + 1] - cu_k[b];
    if (nq < 0 || nk < 0) return SAGE_ERR_INVALID_ARG;
    if (nq > kMaxTokens || nk > kMaxTokens) return SAGE_ERR_UNSUPPORTED;
    if (nq > 0 && nk == 0) return SAGE_ERR_INVALID_ARG;
    if (causal && nq > nk) return SAGE_ERR_UNSUPPORTED;
    P->seqs[b] = VarSeq{(int)nq, (int)nk, cu_q[b], cu_k[b]};
    max_q = std::max(max_q, (int)nq);
    max_k = std::max(max_k, (int)nk);
  }
  if (max_q == 0) return SAGE_ERR_INVALID_ARG;  // nothing to attend
  P->shape = sage_shape{nseq, Hq, Hkv, max_q, max_k, d};
  sage_status st = compute_layout(&P->shape, mode, bq, bk, &P->L);
  if (st != SAGE_OK) return st;
  const int Tm = P->L.Tm;
  std::vector<std::pair<int, int>> work;  // (key tiles, code)
  for (int b = 0; b < nseq; ++b) {
    const VarSeq &q = P->seqs[b];
    const int tm = (int)cdiv(q.N, 128), tn = (int)cdiv(q.M, bk);
    for (int h = 0; h < Hq; ++h)
      for (int i = 0; i < tm; ++i) {
        const int last_row = std::min(q.N, i * 128 + 128) - 1;
        const int T = causal ? std::min(tn, (last_row + q.M - q.N) / bk + 1) : tn;
        work.emplace_back(T, (b * Hq + h) * Tm + i);
      }
  }
  std::stable_sort(work.begin(), work.end(), [](const std::pair<int, int> &x, const std::pair<int, int> &y) {
    return x.first > y.first;
  });
  if (work.size() >= ((size_t)1 << 31)) return SAGE_ERR_UNSUPPORTED;
  P->items = (int)work.size();
  P->item_codes.resize(work.size());
  for (size_t i = 0; i < work.size(); ++i) P->item_codes[i] = work[i].second;
  P->seq_off = P->L.total;
  P->item_off = align_up(P->seq_off + sizeof(VarSeq) * (size_t)nseq, 1024);
  P->total = align_up(P->item_off + sizeof(int) * work.size() + 4, 1024);
  return SAGE_OK;
}

inline StatsView stats_view(void *ws, const sage_ws_layout &L, const sage_shape &s) {
  const size_t n = (size_t)s.B * s.Hkv * s.d;
  char *base = (char *)ws + L.stats;
  StatsView v;
  v.ksum = (int64_t *)base;
  v.vsum = (int64_t *)(base + n * 8);
  v.vmin = (int *)(base + n * 16);
  v.vmax = (int *)(base + n * 20);
  return v;
}

}  // namespace sage
