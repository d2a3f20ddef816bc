"""CPU oracle for the packed (bi)LSTM -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU baseline may
import this package.  The product path (``padding_free_variable_gb300``) never
does, and it shares no code with it.

``lstm_oracle.c`` holds the arithmetic (fp64, one sequence at a time); this
module marshals numpy arrays into it.  ``mdlstm_oracle.c`` / ``mdlstm.py`` do the
same for the 2-D MDLSTM layer, and ``mdlstm.py`` restates the 2-D packing
algorithm.  ``padding.py`` holds the zero-padding
statistics.  Parity status of each function is stated in its docstring.
"""
from .oracle import (  # noqa: F401
    build,
    lstm_stack,
    lstm_padded_layer,
    pack_layer_params,
    round_bf16,
    unpack_layer_grads,
)
from .padding import zero_padding_rate, waste_fraction, bucket_batches  # noqa: F401
from .mdlstm import example_pack, md_layer, md_param_count  # noqa: F401
