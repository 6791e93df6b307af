// bq_multi_q4_k_r56.cu -- Q4_K instances of the multi-op streaming kernel:
// verify with R = 5, 6 (one weight row per lane).
#include "bq_multi_launch.cuh"

BQ_MULTI_UNIT(q4_k, bq::QT_Q4_K, r56,
              BQ_INST(bq::QT_Q4_K, 1, 5),
              BQ_INST(bq::QT_Q4_K, 1, 6))
