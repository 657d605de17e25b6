"""The input generator's chunked form gives exactly the values of its one-shot form."""
import numpy as np

import synth


def test_chunked_inputs_equal_make_inputs():
    w = synth.BY_NAME["mamba130m"].resized(batch=2, T=37, d_inner=50, d_state=12, name="chunks")
    ref = synth.make_inputs(w, seed=3)
    got = {k: np.full(ref[k].size, np.nan, dtype=np.float32) for k in synth.CHUNKED_KEYS}
    pieces = 0
    for name, start, v in synth.iter_input_chunks(w, seed=3, chunk=1000):   # ragged last pieces
        got[name][start:start + v.size] = v
        pieces += 1
    assert pieces > len(synth.CHUNKED_KEYS)
    for k in synth.CHUNKED_KEYS:
        assert np.array_equal(got[k].reshape(ref[k].shape), ref[k]), k
    small = synth.small_inputs(w, seed=3)
    for k in ("A_log", "D"):
        assert np.array_equal(small[k], ref[k]), k
