// bq_multi_q8_0_r56.cu -- Q8_0 instances of the multi-op streaming kernel:
// verify with R = 5, 6 (NR = 1, 2).
#include "bq_multi_launch.cuh"

BQ_MULTI_UNIT(q8_0, bq::QT_Q8_0, r56,
              BQ_INST(bq::QT_Q8_0, 1, 5),
              BQ_INST(bq::QT_Q8_0, 2, 5),
              BQ_INST(bq::QT_Q8_0, 1, 6),
              BQ_INST(bq::QT_Q8_0, 2, 6))
