// bqe_verify.cu — bookkeeping of a speculative verify pass (host code).
//
// The DeepSeek-V4.1-Flash field report (section 3B) decodes with a draft-
// and-verify loop and reports tokens per pass; the 2 x RTX PRO 6000 post
// verifies all candidates layer by layer in one batch, commits the accepted
// prefix and rolls the rejected tail back.  The decode layer computes all
// verify rows in one call (M = drafts + 1); this is the part around it:
// greedy acceptance (a draft is kept while it equals the target's prediction
// at the row before it), the rows to commit, the tokens the pass emits, and
// the statistics (passes, tokens, accepted-length histogram).
#include <stdint.h>

#include "../../include/bqe.h"

extern "C" int bqe_verify_pass(int32_t n_draft, const int32_t* draft, const int32_t* target, int32_t* emitted,
                               int32_t* n_emitted, int32_t* commit_mask, bqe_verify_stats* stats) {
  if (n_draft < 0 || n_draft > BQE_VERIFY_MAX_DRAFT || (n_draft > 0 && !draft) || !target || !emitted ||
      !n_emitted || !commit_mask)
    return BQE_EINVAL;
  int32_t a = 0;
  while (a < n_draft && draft[a] == target[a]) ++a;
  for (int32_t i = 0; i < a; ++i) emitted[i] = draft[i];
  emitted[a] = target[a];  // the target's own token after the last accepted row
  *n_emitted = a + 1;
  for (int32_t r = 0; r <= n_draft; ++r) commit_mask[r] = r <= a ? 1 : 0;
  if (stats) {
    stats->passes += 1;
    stats->tokens += (uint64_t)(a + 1);
    stats->hist[a] += 1;
  }
  return BQE_OK;
}
