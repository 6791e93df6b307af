// bq_gemv_q4_k.cu -- Q4_K: generic kernel, stream executor, multi-op dispatch
// and the format's device error word (bq_format_unit.cuh).
#include "bq_format_unit.cuh"

BQ_FORMAT_UNIT(q4_k, bq::QT_Q4_K)
