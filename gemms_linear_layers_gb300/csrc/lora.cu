// lora.cu -- rank-16 LoRA streaming kernels (see tg_internal.h).
#include "tg_internal.h"
