"""CPU oracle -- test infrastructure only.

Imported by the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline / reference arm, and by
nothing on the product path. It shares no code with the CUDA library (see ``oracle/ref.py``).
"""
from .ref import (attend, chunk_frames, kept_pairs, kept_set_of_frame, kept_set_of_global, num_chunks,  # noqa: F401
                  row_logsumexp, window_attention, window_attention_backward, window_attention_backward_rows,
                  window_attention_rows)
