// KDA oracle: a plain, slow, double-precision CPU restatement of the Kimi Delta Attention
// (KDA) gated delta-rule recurrence and of the segment-package algebra built on it.
//
// TEST INFRASTRUCTURE ONLY. This file is used by the test-suite, by the smoke check and by
// the benchmark's CPU-baseline leg. The product library never links, loads or calls it, and
// it shares no code, header, table or constant with the CUDA path.
//
// What is computed (per sequence, per head; S has dk rows and dv columns, row = key channel):
//   S_t = (I - beta_t k_t k_t^T) Diag(a_t) S_{t-1} + beta_t k_t v_t^T,  a_t = exp(g_t),
//   o_t = scale * S_t^T q_t.
// The recurrence is the one the pegainfer pull request #970 ("feat(k3): cross-process CP
// whale gang - fleet-wide long-prompt prefill") prefills with FlashKDA and publishes as one
// KDA (M,D) package per context-parallel segment (commit message of the fabric data-plane
// change); the pages name the operator but do not write the formula, so the formula above is
// the plainest statement of the gated delta rule with per-key-channel decay, decay applied
// before the erase, and the output read from the updated state.
//
// It is evaluated in the algebraically identical "delta" order, one token at a time:
//   S <- Diag(a_t) S;  u = v_t - S^T k_t;  S <- S + beta_t k_t u^T;  o_t = scale S^T q_t.
// (Expand (I - b k k^T) D S + b k v^T = D S + b k (v - (D S)^T k)^T.)
//
// Segment packages ((M,D) packages of the same page): a token range maps any entry state
// S_in to S_out = M S_in + D. Running the recurrence on the augmented dk x (dk+dv) state
// [M | D] from [I | 0] with values [0 | v] yields exactly that pair, because the columns of
// S evolve independently and linearly in (S, v). Packages compose with
//   (M2, D2) o (M1, D1) = (M2 M1, M2 D1 + D2),
// and a segmented exclusive prefix over the packages gives each segment its entry state.
//
// Every loop runs in the order written, in double precision, with no blocking, fusion or
// reordering. Threads split independent (sequence, head, column-block) work items only;
// the arithmetic on each item is the same single-threaded loop.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <atomic>
#include <thread>
#include <vector>
#include <algorithm>

namespace {

// Runs fn(item) for item in [0, n_items) on up to n_threads threads (0 => hardware count).
template <class F>
int parallel_items(int64_t n_items, int n_threads, F fn) {
  if (n_threads <= 0) {
    n_threads = (int)std::thread::hardware_concurrency();
    if (n_threads <= 0) n_threads = 1;
  }
  if ((int64_t)n_threads > n_items) n_threads = (int)std::max<int64_t>(n_items, 1);
  std::atomic<int64_t> next(0);
  auto worker = [&]() {
    for (;;) {
      int64_t it = next.fetch_add(1);
      if (it >= n_items) break;
      fn(it);
    }
  };
  if (n_threads == 1) {
    worker();
  } else {
    std::vector<std::thread> pool;
    for (int i = 0; i < n_threads; ++i) pool.emplace_back(worker);
    for (auto& t : pool) t.join();
  }
  return n_threads;
}

// One column block of the recurrence for one (sequence, head) over tokens [t0, t1).
// S is dk x ncols (row-major, ncols = j1 - j0) holding columns [j0, j1) of the full state.
// vcol(t, j) returns the value entry for token t, full-state column j.
// Layouts: x[t][h][c] with strides H*dx and dx.
template <class VCol>
void recur_block(int t0, int t1, int h, int H, int dk, int j0, int j1, double scale,
                 const double* q, const double* k, const double* g, const double* beta,
                 VCol vcol, double* S, double* o, int o_stride_t, int o_col_offset) {
  const int nc = j1 - j0;
  std::vector<double> a(dk), kt(dk), u(nc);
  for (int t = t0; t < t1; ++t) {
    const double* kk = k + ((int64_t)t * H + h) * dk;
    const double* gg = g + ((int64_t)t * H + h) * dk;
    const double b = beta[(int64_t)t * H + h];
    for (int c = 0; c < dk; ++c) a[c] = std::exp(gg[c]);
    // decay: S <- Diag(a) S
    for (int c = 0; c < dk; ++c)
      for (int j = 0; j < nc; ++j) S[(int64_t)c * nc + j] *= a[c];
    // prediction error: u = v - S^T k
    for (int j = 0; j < nc; ++j) {
      double acc = 0.0;
      for (int c = 0; c < dk; ++c) acc += kk[c] * S[(int64_t)c * nc + j];
      u[j] = vcol(t, j0 + j) - acc;
    }
    // write: S <- S + beta k u^T
    for (int c = 0; c < dk; ++c)
      for (int j = 0; j < nc; ++j) S[(int64_t)c * nc + j] += b * kk[c] * u[j];
    // read: o = scale S^T q
    if (o) {
      const double* qq = q + ((int64_t)t * H + h) * dk;
      for (int j = 0; j < nc; ++j) {
        double acc = 0.0;
        for (int c = 0; c < dk; ++c) acc += qq[c] * S[(int64_t)c * nc + j];
        o[(int64_t)t * o_stride_t + o_col_offset + j] = scale * acc;
      }
    }
  }
}

constexpr int kColBlock = 32;

}  // namespace

extern "C" {

// Sequential pass over packed sequences.
//   cu_seqlens: [n_seqs+1] token offsets (cu_seqlens[0] = 0, non-decreasing).
//   q, k, g: [T, H, dk]; v: [T, H, dv]; beta: [T, H]; init_state: [n_seqs, H, dk, dv] or NULL
//   (zeros). Outputs o: [T, H, dv] (may be NULL), final_state: [n_seqs, H, dk, dv] (may be
//   NULL). Returns the number of threads used, or -1 on bad arguments.
int kda_ref_forward(int n_seqs, const int64_t* cu_seqlens, int H, int dk, int dv, double scale,
                    const double* q, const double* k, const double* v, const double* g,
                    const double* beta, const double* init_state, double* o,
                    double* final_state, int n_threads) {
  if (n_seqs < 0 || H <= 0 || dk <= 0 || dv <= 0 || !cu_seqlens) return -1;
  const int nblk = (dv + kColBlock - 1) / kColBlock;
  const int64_t n_items = (int64_t)n_seqs * H * nblk;
  return parallel_items(n_items, n_threads, [&](int64_t it) {
    const int blk = (int)(it % nblk);
    const int h = (int)((it / nblk) % H);
    const int s = (int)(it / ((int64_t)nblk * H));
    const int j0 = blk * kColBlock, j1 = std::min(dv, j0 + kColBlock), nc = j1 - j0;
    std::vector<double> S((size_t)dk * nc, 0.0);
    if (init_state) {
      const double* S0 = init_state + ((int64_t)s * H + h) * dk * dv;
      for (int c = 0; c < dk; ++c)
        for (int j = 0; j < nc; ++j) S[(size_t)c * nc + j] = S0[(int64_t)c * dv + j0 + j];
    }
    auto vcol = [&](int t, int j) { return v[((int64_t)t * H + h) * dv + j]; };
    double* ob = o ? o + (int64_t)h * dv : nullptr;
    recur_block((int)cu_seqlens[s], (int)cu_seqlens[s + 1], h, H, dk, j0, j1, scale, q, k, g,
                beta, vcol, S.data(), ob, H * dv, j0);
    if (final_state) {
      double* SF = final_state + ((int64_t)s * H + h) * dk * dv;
      for (int c = 0; c < dk; ++c)
        for (int j = 0; j < nc; ++j) SF[(int64_t)c * dv + j0 + j] = S[(size_t)c * nc + j];
    }
  });
}

// Segment packages: for each segment [seg_offsets[p], seg_offsets[p+1]) and head, the pair
// (M, D) with S_out = M S_in + D for any entry state S_in.
//   M: [n_segs, H, dk, dk]; D: [n_segs, H, dk, dv]. Returns threads used, or -1.
int kda_ref_package(int n_segs, const int64_t* seg_offsets, int H, int dk, int dv,
                    const double* k, const double* v, const double* g, const double* beta,
                    double* M, double* D, int n_threads) {
  if (n_segs < 0 || H <= 0 || dk <= 0 || dv <= 0 || !seg_offsets || !M || !D) return -1;
  const int width = dk + dv;  // augmented state [M | D]
  const int nblk = (width + kColBlock - 1) / kColBlock;
  const int64_t n_items = (int64_t)n_segs * H * nblk;
  return parallel_items(n_items, n_threads, [&](int64_t it) {
    const int blk = (int)(it % nblk);
    const int h = (int)((it / nblk) % H);
    const int p = (int)(it / ((int64_t)nblk * H));
    const int j0 = blk * kColBlock, j1 = std::min(width, j0 + kColBlock), nc = j1 - j0;
    // entry [I | 0]
    std::vector<double> S((size_t)dk * nc, 0.0);
    for (int c = 0; c < dk; ++c)
      for (int j = 0; j < nc; ++j) S[(size_t)c * nc + j] = (j0 + j == c) ? 1.0 : 0.0;
    // values [0 | v]
    auto vcol = [&](int t, int j) {
      return j < dk ? 0.0 : v[((int64_t)t * H + h) * dv + (j - dk)];
    };
    recur_block((int)seg_offsets[p], (int)seg_offsets[p + 1], h, H, dk, j0, j1, 1.0, nullptr,
                k, g, beta, vcol, S.data(), nullptr, 0, 0);
    double* Mp = M + ((int64_t)p * H + h) * dk * dk;
    double* Dp = D + ((int64_t)p * H + h) * dk * dv;
    for (int c = 0; c < dk; ++c)
      for (int j = 0; j < nc; ++j) {
        const int col = j0 + j;
        if (col < dk) Mp[(int64_t)c * dk + col] = S[(size_t)c * nc + j];
        else Dp[(int64_t)c * dv + (col - dk)] = S[(size_t)c * nc + j];
      }
  });
}

// Composition of two packages of one head: (M, D) = (M2, D2) o (M1, D1)
//   = (M2 M1, M2 D1 + D2); M* are dk x dk, D* are dk x dv, all row-major.
void kda_ref_compose(int dk, int dv, const double* M2, const double* D2, const double* M1,
                     const double* D1, double* M, double* D) {
  for (int r = 0; r < dk; ++r) {
    for (int c = 0; c < dk; ++c) {
      double acc = 0.0;
      for (int x = 0; x < dk; ++x) acc += M2[(int64_t)r * dk + x] * M1[(int64_t)x * dk + c];
      M[(int64_t)r * dk + c] = acc;
    }
    for (int c = 0; c < dv; ++c) {
      double acc = D2[(int64_t)r * dv + c];
      for (int x = 0; x < dk; ++x) acc += M2[(int64_t)r * dk + x] * D1[(int64_t)x * dv + c];
      D[(int64_t)r * dv + c] = acc;
    }
  }
}

// Segmented exclusive prefix over packages, as a sequential left fold per (sequence, head):
// segments [seq_seg_offsets[s], seq_seg_offsets[s+1]) belong to sequence s, in token order.
//   seg_init[first] = init_state[s] (zeros if NULL); seg_init[j+1] = M_j seg_init[j] + D_j;
//   final_state[s] = M_last seg_init[last] + D_last (init_state[s] if s has no segments).
// seg_init: [n_segs, H, dk, dv]; final_state: [n_seqs, H, dk, dv] or NULL.
int kda_ref_scan(int n_seqs, const int64_t* seq_seg_offsets, int H, int dk, int dv,
                 const double* M, const double* D, const double* init_state, double* seg_init,
                 double* final_state, int n_threads) {
  if (n_seqs < 0 || H <= 0 || dk <= 0 || dv <= 0 || !seq_seg_offsets || !seg_init) return -1;
  const int64_t n_items = (int64_t)n_seqs * H;
  return parallel_items(n_items, n_threads, [&](int64_t it) {
    const int h = (int)(it % H);
    const int s = (int)(it / H);
    const int64_t sd = (int64_t)dk * dv;
    std::vector<double> cur(sd, 0.0), nxt(sd);
    if (init_state) std::memcpy(cur.data(), init_state + ((int64_t)s * H + h) * sd, sd * 8);
    for (int64_t p = seq_seg_offsets[s]; p < seq_seg_offsets[s + 1]; ++p) {
      std::memcpy(seg_init + (p * H + h) * sd, cur.data(), sd * 8);
      const double* Mp = M + (p * H + h) * (int64_t)dk * dk;
      const double* Dp = D + (p * H + h) * sd;
      for (int r = 0; r < dk; ++r)
        for (int c = 0; c < dv; ++c) {
          double acc = Dp[(int64_t)r * dv + c];
          for (int x = 0; x < dk; ++x) acc += Mp[(int64_t)r * dk + x] * cur[(int64_t)x * dv + c];
          nxt[(int64_t)r * dv + c] = acc;
        }
      cur.swap(nxt);
    }
    if (final_state) std::memcpy(final_state + ((int64_t)s * H + h) * sd, cur.data(), sd * 8);
  });
}

// One decode token per batch row over a slot-addressed state pool, updated in place.
//   q, k, g: [B, H, dk]; v: [B, H, dv]; beta: [B, H]; slot_ids: [B];
//   pool: [n_slots, H, dk, dv]. A row whose slot id is negative (padding) or >= n_slots is
//   skipped and its output row is zero. Returns the number of out-of-range (>= n_slots)
//   slot ids seen, or -1 on bad arguments.
int kda_ref_decode(int B, int H, int dk, int dv, double scale, const double* q,
                   const double* k, const double* v, const double* g, const double* beta,
                   const int64_t* slot_ids, double* pool, int64_t n_slots, double* o,
                   int n_threads) {
  if (B < 0 || H <= 0 || dk <= 0 || dv <= 0 || !slot_ids || !pool || !o) return -1;
  std::atomic<int> bad(0);
  parallel_items((int64_t)B * H, n_threads, [&](int64_t it) {
    const int h = (int)(it % H);
    const int b = (int)(it / H);
    const int64_t s = slot_ids[b];
    double* ob = o + ((int64_t)b * H + h) * dv;
    if (s < 0 || s >= n_slots) {
      if (s >= n_slots && h == 0) bad.fetch_add(1);
      for (int j = 0; j < dv; ++j) ob[j] = 0.0;
      return;
    }
    double* S = pool + (s * H + h) * (int64_t)dk * dv;
    auto vcol = [&](int, int j) { return v[((int64_t)b * H + h) * dv + j]; };
    // one token (row b of the batch arrays) on the block holding all dv columns
    recur_block(b, b + 1, h, H, dk, 0, dv, scale, q, k, g, beta, vcol, S, o, H * dv, h * dv);
  });
  return bad.load();
}

// A verify window of W tokens per batch row, with a state fork: for row b and head h the
// state is read from slot read_slots[b] and, after each token j of the row's window, the
// current state is stored into slot write_slots[b*W + j] (a per-column snapshot, so that a
// caller that accepts only the first n tokens resumes from the snapshot of column n - 1).
// This is the read/write state-index split of ATOM PR #2709 ("feat(kimi-k3): PP8 prefill for
// P/D serving - KDA state under PP"): a forked state is read through a read-side slot index,
// and a verify window keeps one state column per position, the next step starting from the
// last accepted one. The recurrence per token is exactly the one above.
//   q, k, g: [B*W, H, dk]; v: [B*W, H, dv]; beta: [B*W, H] (token b*W + j is column j of row
//   b); read_slots: [B]; write_slots: [B*W]; pool: [n_slots, H, dk, dv]; o: [B*W, H, dv].
//   beta_is_logit != 0: beta holds logits and the write strength is 1 / (1 + exp(-beta)).
// A row whose read slot is negative (padding) or >= n_slots is skipped: its outputs are zero
// and nothing is stored. A negative write slot stores nothing for that column; one >= n_slots
// is skipped and counted. Returns the number of out-of-range slot ids seen (each counted
// once, on head 0), or -1 on bad arguments.
int kda_ref_decode_window(int B, int W, int H, int dk, int dv, double scale, const double* q,
                          const double* k, const double* v, const double* g,
                          const double* beta, int beta_is_logit, const int64_t* read_slots,
                          const int64_t* write_slots, double* pool, int64_t n_slots,
                          double* o, int n_threads) {
  if (B < 0 || W < 0 || H <= 0 || dk <= 0 || dv <= 0 || !read_slots || !write_slots || !pool ||
      !o)
    return -1;
  // write strengths of every (token, head), from the logits where asked
  const int64_t n_tok = (int64_t)B * W;
  std::vector<double> bw((size_t)(n_tok * H));
  for (int64_t i = 0; i < n_tok * H; ++i)
    bw[i] = beta_is_logit ? 1.0 / (1.0 + std::exp(-beta[i])) : beta[i];
  std::atomic<int> bad(0);
  const int64_t sd = (int64_t)dk * dv;
  parallel_items((int64_t)B * H, n_threads, [&](int64_t it) {
    const int h = (int)(it % H);
    const int b = (int)(it / H);
    const int64_t r = read_slots[b];
    if (r < 0 || r >= n_slots) {
      if (r >= n_slots && h == 0) bad.fetch_add(1);
      for (int j = 0; j < W; ++j)
        for (int c = 0; c < dv; ++c) o[(((int64_t)b * W + j) * H + h) * dv + c] = 0.0;
      return;
    }
    std::vector<double> S(pool + (r * H + h) * sd, pool + (r * H + h) * sd + sd);
    auto vcol = [&](int t, int c) { return v[((int64_t)t * H + h) * dv + c]; };
    for (int j = 0; j < W; ++j) {
      const int t = b * W + j;
      recur_block(t, t + 1, h, H, dk, 0, dv, scale, q, k, g, bw.data(), vcol, S.data(), o,
                  H * dv, h * dv);
      const int64_t w = write_slots[t];
      if (w >= n_slots) {
        if (h == 0) bad.fetch_add(1);
      } else if (w >= 0) {
        std::memcpy(pool + (w * H + h) * sd, S.data(), sd * sizeof(double));
      }
    }
  });
  return bad.load();
}

// Short causal depthwise convolution over packed varlen rows, with a per-sequence window of
// the last (W - 1) inputs kept in a slot pool: the KDA short-conv gather and window update of
// kern PR #44 (per-sequence varlen kernels of the stage split), read through a read-side slot
// index as in ATOM PR #2709 (the spec conv update takes a read index). The pages do not give
// the width W or an activation; both are parameters here.
// For sequence s and channel c, with history h (W - 1 inputs, oldest first) taken from slot
// read_slots[s] (zeros when the id is negative or read_slots is NULL):
//   y_t = sum_{i=0}^{W-1} w[c, i] * z[t - (W - 1) + i],  z = [h ; x_s]  (w[c, W-1] multiplies
//   the current input), out_t = silu ? y_t / (1 + exp(-y_t)) : y_t,
// and afterwards the last W - 1 entries of z are stored into slot write_slots[s] (not stored
// when the id is negative or write_slots is NULL).
//   cu_seqlens: [n_seqs+1]; x, out: [T, C]; w: [C, W]; pool: [n_slots, W-1, C].
// Ids >= n_slots are skipped (read: zero history; write: nothing stored) and counted.
// Returns the count, or -1 on bad arguments.
int kda_ref_short_conv(int n_seqs, const int64_t* cu_seqlens, int C, int W, const double* x,
                       const double* w, int silu, const int64_t* read_slots,
                       const int64_t* write_slots, double* pool, int64_t n_slots, double* out,
                       int n_threads) {
  if (n_seqs < 0 || C <= 0 || W <= 0 || !cu_seqlens || !x || !w || !out) return -1;
  if ((read_slots || write_slots) && !pool) return -1;
  std::atomic<int> bad(0);
  const int nblk = (C + kColBlock - 1) / kColBlock;
  const int hw = W - 1;
  parallel_items((int64_t)n_seqs * nblk, n_threads, [&](int64_t it) {
    const int blk = (int)(it % nblk);
    const int s = (int)(it / nblk);
    const int c0 = blk * kColBlock, c1 = std::min(C, c0 + kColBlock);
    const int64_t r = read_slots ? read_slots[s] : -1;
    const int64_t wr = write_slots ? write_slots[s] : -1;
    if (blk == 0) bad.fetch_add((r >= n_slots ? 1 : 0) + (wr >= n_slots ? 1 : 0));
    const int64_t t0 = cu_seqlens[s], t1 = cu_seqlens[s + 1];
    for (int c = c0; c < c1; ++c) {
      // z = [h ; x_s] for this channel
      std::vector<double> z((size_t)(hw + (t1 - t0)), 0.0);
      if (r >= 0 && r < n_slots)
        for (int j = 0; j < hw; ++j) z[j] = pool[(r * hw + j) * C + c];
      for (int64_t t = t0; t < t1; ++t) z[hw + (t - t0)] = x[t * C + c];
      for (int64_t t = t0; t < t1; ++t) {
        const int64_t u = hw + (t - t0);  // position of x_t in z
        double y = 0.0;
        for (int i = 0; i < W; ++i) y += w[(int64_t)c * W + i] * z[u - hw + i];
        out[t * C + c] = silu ? y / (1.0 + std::exp(-y)) : y;
      }
      if (wr >= 0 && wr < n_slots) {
        const size_t n = z.size();
        for (int j = 0; j < hw; ++j) pool[(wr * hw + j) * C + c] = z[n - hw + j];
      }
    }
  });
  return bad.load();
}

}  // extern "C"
