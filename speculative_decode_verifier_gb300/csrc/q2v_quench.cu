// q2v_quench.cu -- the terminal yield-quench controller: a host-side consumer of the verify's
// accepted counts ("ds4-on-spark" README, "The break-even law"; "1x Spark tuned DSpark ...",
// "The break-even law, and why speculation can't hurt you here").
//
// One verify step costs about `guard` plain decode steps (2.16 for the current weights) and
// commits n_accepted + 1 tokens.  Each step adds the regret guard - (n_accepted + 1) to the
// session's running total; once the total exceeds `threshold` plain-step times (about 4),
// speculation is switched off for the rest of that request.  Plain host code, no CUDA.
#include <math.h>
#include <stddef.h>

#include "../../include/q2v.h"

extern "C" {

q2_status q2_quench_init(q2_quench_state *state, int S) {
    if (!state || S < 1) return Q2_ERR_INVALID_ARG;
    for (int s = 0; s < S; ++s) {
        state[s].regret = 0.0;
        state[s].steps = 0;
        state[s].quenched = 0;
    }
    return Q2_OK;
}

int q2_quench_update(q2_quench_state *state, int S, const int32_t *n_accepted, double guard,
                     double threshold) {
    if (!state || !n_accepted || S < 1 || !isfinite(guard) || !isfinite(threshold)) return -1;
    int newly = 0;
    for (int s = 0; s < S; ++s) {
        q2_quench_state &q = state[s];
        if (q.quenched || n_accepted[s] < 0) continue;  // quenched for good; a bad session's step is skipped
        q.regret += guard - (double)(n_accepted[s] + 1);
        ++q.steps;
        if (q.regret > threshold) {
            q.quenched = 1;
            ++newly;
        }
    }
    return newly;
}

}  // extern "C"
