// bq_multi_q4_0_r56.cu -- Q4_0 instances of the multi-op streaming kernel:
// verify with R = 5, 6 (NR = 1, 2).
#include "bq_multi_launch.cuh"

BQ_MULTI_UNIT(q4_0, bq::QT_Q4_0, r56,
              BQ_INST(bq::QT_Q4_0, 1, 5),
              BQ_INST(bq::QT_Q4_0, 2, 5),
              BQ_INST(bq::QT_Q4_0, 1, 6),
              BQ_INST(bq::QT_Q4_0, 2, 6))
