// prefill_masked.cu -- the prefill kernels with an explicit attention mask: the same kernel
// template as prefill.cu, instantiated with MASK = true (paged pool) in a translation unit of its own.
#define ASTR_PREFILL_MASKED_TU 1
#include "prefill.cu"
