"""The replay bundle a failed parity case leaves (host side, no GPU)."""
import hashlib
import json

import numpy as np

import datagen
import parity


def test_replay_bundle_identifies_the_case(tmp_path):
    """A failed parity case leaves a bundle that names the workload and the
    exact inputs (SHA-256 of the bits and of the fp32 parameters)."""
    wl = datagen.WORKLOADS["tiny_diag"].with_n(300)
    mix = datagen.planted(wl)
    bits = datagen.points(mix, 0, wl.N)
    theta = tuple(np.asarray(p, dtype=np.float32) for p in datagen.init_params(mix, bits))
    path = parity.replay_bundle(wl, bits, theta, ["mu[3]: rel err 5e-3"], str(tmp_path))
    rec = json.load(open(path))
    assert (rec["workload"], rec["N"], rec["D"], rec["K"]) == ("tiny_diag", 300, wl.D, wl.K)
    assert rec["x_sha256"] == hashlib.sha256(np.ascontiguousarray(bits).tobytes()).hexdigest()
    assert rec["params_sha256"][1] == hashlib.sha256(theta[1].tobytes()).hexdigest()
    assert rec["failures"] == ["mu[3]: rel err 5e-3"]
    # the same inputs give the same digests (the bundle identifies them)
    bits2 = datagen.points(mix, 0, wl.N)
    assert hashlib.sha256(np.ascontiguousarray(bits2).tobytes()).hexdigest() == rec["x_sha256"]
    # a directory that cannot be made does not raise
    blocker = tmp_path / "file"
    blocker.write_text("x")
    assert parity.replay_bundle(wl, bits, theta, [], str(blocker / "sub")) is None
