"""CPU oracle (test infrastructure only): plain fp64 restatement of the method."""
