// Tensor-core window scoring (tcgen05 + TMA + TMEM) for bf16 keys.
#include "common.cuh"

namespace chunkkv {

bool tc_supported(const Plan& pl) { (void)pl; return false; }

void tc_plan(Plan& pl) { pl.use_tc = 0; pl.tc_mt = 0; }

cudaError_t launch_score_tc(const Plan& pl, const ScoreGeom& g, const SeqTable& st, const void* q,
                            const void* k, float* rl, float* bins, void* qpack, int32_t* err,
                            cudaStream_t s) {
  (void)pl; (void)g; (void)st; (void)q; (void)k; (void)rl; (void)bins; (void)qpack; (void)err; (void)s;
  return cudaErrorNotSupported;
}

}  // namespace chunkkv
