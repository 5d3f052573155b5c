"""Records the parity figures of GPU tests (code mismatch against the float32 and
float64 oracle, dequantized weights off the float64 oracle's by more than half a step,
scale error, output error) as JSON lines in the file named by the environment variable
GPTQ_PARITY_LOG, when it is set. Test infrastructure only."""
import json
import os


def record(case: str, **figures) -> None:
    path = os.environ.get("GPTQ_PARITY_LOG")
    if not path:
        return
    row = {"case": case}
    for k, v in figures.items():
        row[k] = float(v) if hasattr(v, "__float__") else v
    with open(path, "a") as f:
        f.write(json.dumps(row) + "\n")
