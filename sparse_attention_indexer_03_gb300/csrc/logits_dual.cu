// The tensor-core logits kernel instantiated with two MMA warps (decode-like
// shapes on pages of 64 tokens or more), in a translation unit of its own so
// that it compiles in parallel with the other instantiations.
#define SAI_LOGITS_DUAL 1
#include "logits.cu"
