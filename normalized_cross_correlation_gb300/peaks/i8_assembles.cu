// i8_assembles.cu -- compile-only check: does ptxas accept an integer
// tcgen05.mma (kind::i8, s8/u8 operands, s32 accumulator) for a target?  The
// runner assembles this file for sm_103a and for sm_100a and reports which
// succeed.  Nothing here is launched.
#include <cstdint>

__global__ void i8_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc) {
    asm volatile("{ .reg .pred p; setp.ne.b32 p, %4, 0;\n"
                 "tcgen05.mma.cta_group::1.kind::i8 [%0], %1, %2, %3, p; }"
                 ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(1u) : "memory");
}
