// bq_gemv_q4_0.cu -- Q4_0: generic kernel, stream executor, multi-op dispatch
// and the format's device error word (bq_format_unit.cuh).
#include "bq_format_unit.cuh"

BQ_FORMAT_UNIT(q4_0, bq::QT_Q4_0)
