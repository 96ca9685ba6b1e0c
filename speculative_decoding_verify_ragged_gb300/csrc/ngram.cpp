// n-gram (prompt-lookup) drafting on the host (declared in sdv_draft.h).
//
// Copy-style drafting needs no draft model: the longest recent suffix of a
// sequence that already occurred earlier in it is assumed to continue the way
// it did then (splicedso primer on speculative decoding, section "When it
// works": n-gram drafting copies text already in the prompt).  The search runs
// from the most recent earlier position backwards, so the first match is the
// most recent occurrence; longer suffixes are tried first.
#include <cstring>

#include "sdv_draft.h"

namespace {

// Does history[i .. i + n) equal the last n tokens?
bool matches_suffix(const int* h, int len, int i, int n) {
  return std::memcmp(h + i, h + len - n, sizeof(int) * static_cast<size_t>(n)) == 0;
}

int draft_one(const int* h, int len, int min_n, int max_n, int gamma, int* out) {
  if (gamma <= 0) return 0;
  for (int n = max_n < len - 1 ? max_n : len - 1; n >= min_n; --n) {
    // an earlier occurrence must leave at least one token after it
    for (int i = len - n - 1; i >= 0; --i) {
      if (!matches_suffix(h, len, i, n)) continue;
      const int start = i + n;
      int k = len - start;
      if (k > gamma) k = gamma;
      for (int j = 0; j < k; ++j) out[j] = h[start + j];
      return k;
    }
  }
  return 0;
}

}  // namespace

extern "C" {

int sdv_ngram_draft(const int* history, int len, int min_n, int max_n, int gamma, int* drafts) {
  if (len < 0 || min_n < 1 || max_n < min_n || gamma < 0) return -1;
  if ((len > 0 && !history) || (gamma > 0 && !drafts)) return -1;
  return draft_one(history, len, min_n, max_n, gamma, drafts);
}

sdv_status sdv_ngram_draft_batch(const int* tokens, const long long* offsets, int B, int min_n, int max_n,
                                 int gamma_max, int* draft_lens, int* drafts) {
  if (B < 0 || !offsets || min_n < 1 || max_n < min_n || gamma_max < 0) return SDV_ERR_INVALID_ARG;
  if (B > 0 && (!draft_lens || (gamma_max > 0 && !drafts))) return SDV_ERR_INVALID_ARG;
  for (int b = 0; b < B; ++b) {
    if (offsets[b] < 0 || offsets[b + 1] < offsets[b]) return SDV_ERR_INVALID_ARG;
    if (offsets[b + 1] > offsets[b] && !tokens) return SDV_ERR_INVALID_ARG;
  }
  for (int b = 0; b < B; ++b) {
    int* row = drafts + static_cast<long long>(b) * gamma_max;
    const int len = static_cast<int>(offsets[b + 1] - offsets[b]);
    const int k = draft_one(tokens + offsets[b], len, min_n, max_n, gamma_max, row);
    for (int j = k; j < gamma_max; ++j) row[j] = -1;
    draft_lens[b] = k;
  }
  return SDV_OK;
}

}  // extern "C"
