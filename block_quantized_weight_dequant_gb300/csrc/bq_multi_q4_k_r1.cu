// bq_multi_q4_k_r1.cu -- Q4_K instances of the multi-op streaming kernel:
// decode and gate+up (R = 1: row mode, NR = 1).
#include "bq_multi_launch.cuh"

BQ_MULTI_UNIT(q4_k, bq::QT_Q4_K, r1,
              BQ_INST(bq::QT_Q4_K, 0, 1),
              BQ_INST(bq::QT_Q4_K, 1, 1))
