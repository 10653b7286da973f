"""Oracle for paged-KV decode attention: plain, slow, fp64, CPU only.

TEST INFRASTRUCTURE. Only tests/, the package entry module's smoke() and
bench.py's cpu_baseline leg may import it. The product path never does.
"""

from . import kv_append  # noqa: F401
from .pa_oracle import (  # noqa: F401
    as_oracle_inputs,
    attend,
    bf16_bits_to_f64,
    combine,
    decode,
    decode_split,
    e4m3fn_table,
    e4m3fn_value,
    f16_bits_to_f64,
    keys_values,
    split_page_ranges,
)
